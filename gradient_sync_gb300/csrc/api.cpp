// C ABI of the all-reduce library: descriptor validation, the schedules' step
// tables (built on the host from the pages' index rules), execution, the
// bucket calls and the host-memory variant.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <mutex>
#include <new>
#include <vector>

#include "internal.h"

using namespace ar;

namespace {

constexpr int kVersion = 1;

bool is_pow2(int n) { return n > 0 && (n & (n - 1)) == 0; }
int64_t imod(int64_t a, int64_t n) { return ((a % n) + n) % n; }
size_t esize(ar_dtype d) { return d == AR_BF16 ? 2 : 4; }
int64_t rup(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
int64_t rdown(int64_t x, int64_t a) { return x / a * a; }

// Cut [lo, hi) into n parts: part p is [lo + p*len/n, lo + (p+1)*len/n).
std::vector<int64_t> cuts(int64_t lo, int64_t hi, int n) {
  std::vector<int64_t> b(n + 1);
  for (int p = 0; p <= n; ++p) b[p] = lo + (int64_t(p) * (hi - lo)) / n;
  return b;
}

Transfer make_xfer(int src, int dst, int64_t lo, int64_t hi, Space xs, Space ys, Space ds, bool fin) {
  Transfer t;
  t.src = int16_t(src);
  t.dst = int16_t(dst);
  t.src2 = -1;
  t.xs = xs;
  t.ys = ys;
  t.ds = ds;
  t.x2s = RAW;
  t.fin = fin ? 1 : 0;
  t.pair = 0;
  t.lo = lo;
  t.hi = hi;
  return t;
}

void add_xfer(Step& st, int src, int dst, int64_t lo, int64_t hi, Space xs, Space ys, Space ds,
              bool fin) {
  if (hi <= lo) return;  // L < N leaves some chunks empty
  st.xfers.push_back(make_xfer(src, dst, lo, hi, xs, ys, ds, fin));
}

// Ring all-reduce (primer ch. 4, "Collective communication: algorithms, cost
// and the library that runs them", §4.2 "The ring, one step at a time").
// Reduce-scatter step s = 0..N-2: rank i sends chunk (i - s) mod N to rank
// i + 1, which adds its own copy; after N-1 steps rank i owns chunk
// (i + 1) mod N. All-gather step s: rank i sends complete chunk
// (i + 1 - s) mod N, which the receiver overwrites.
void build_ring(ar_plan_t* p) {
  const int N = p->desc.n_ranks;
  const int64_t L = int64_t(p->desc.count);
  const auto b = cuts(0, L, N);
  for (int s = 0; s <= N - 2; ++s) {
    Step st{OP_ADD, {}};
    const bool last = s == N - 2;
    for (int i = 0; i < N; ++i) {
      const int c = int(imod(i - s, N));
      add_xfer(st, i, (i + 1) % N, b[c], b[c + 1], s == 0 ? RAW : PART, RAW, last ? RES : PART, last);
    }
    p->steps.push_back(st);
  }
  for (int s = 0; s <= N - 2; ++s) {
    Step st{OP_COPY, {}};
    for (int i = 0; i < N; ++i) {
      const int c = int(imod(i + 1 - s, N));
      add_xfer(st, i, (i + 1) % N, b[c], b[c + 1], RES, RES, RES, false);
    }
    p->steps.push_back(st);
  }
}

// Standalone ring reduce-scatter (primer §4.1 table: each rank ends with S/N
// of the sum). Rank i must end with chunk i, so rank i sends chunk
// (i - 1 - s) mod N at step s (the slice rule of the hierarchical
// reduce-scatter, §4.4); after N-1 steps rank i holds the complete chunk i.
void build_ring_reduce_scatter(ar_plan_t* p) {
  const int N = p->desc.n_ranks;
  const int64_t L = int64_t(p->desc.count);
  const auto b = cuts(0, L, N);
  for (int s = 0; s <= N - 2; ++s) {
    Step st{OP_ADD, {}};
    const bool last = s == N - 2;
    for (int i = 0; i < N; ++i) {
      const int c = int(imod(i - 1 - s, N));
      add_xfer(st, i, (i + 1) % N, b[c], b[c + 1], s == 0 ? RAW : PART, RAW, last ? RES : PART, last);
    }
    p->steps.push_back(st);
  }
}

// Standalone ring all-gather: rank i contributes chunk i and sends chunk
// (i - s) mod N at step s; the receiver overwrites. The first step reads the
// senders' own chunks from the inputs.
void build_ring_allgather(ar_plan_t* p) {
  const int N = p->desc.n_ranks;
  const int64_t L = int64_t(p->desc.count);
  const auto b = cuts(0, L, N);
  for (int s = 0; s <= N - 2; ++s) {
    Step st{OP_COPY, {}};
    for (int i = 0; i < N; ++i) {
      const int c = int(imod(i - s, N));
      add_xfer(st, i, (i + 1) % N, b[c], b[c + 1], s == 0 ? RAW : RES, RES, RES, false);
    }
    p->steps.push_back(st);
  }
}

// Rabenseifner: recursive halving reduce-scatter, recursive doubling
// all-gather (primer §4.3, Fig. 4.5 and Animation 4.2). Step k = 1..log2 N:
// rank i pairs with i xor 2^(k-1), keeps the lower half of its chunk range if
// bit k-1 of i is 0 (else the upper half), sends the other half and adds
// what arrives; the all-gather runs the pairs in reverse order and copies.
void build_rabenseifner(ar_plan_t* p) {
  const int N = p->desc.n_ranks;
  const int64_t L = int64_t(p->desc.count);
  const auto b = cuts(0, L, N);
  int K = 0;
  while ((1 << K) < N) ++K;
  std::vector<std::pair<int, int>> rng(N, {0, N});
  for (int k = 1; k <= K; ++k) {
    const int d = 1 << (k - 1);
    Step st{OP_ADD, {}};
    std::vector<std::pair<int, int>> next(rng);
    for (int i = 0; i < N; ++i) {
      const int lo = rng[i].first, hi = rng[i].second, mid = (lo + hi) / 2;
      const bool lower = ((i >> (k - 1)) & 1) == 0;
      const std::pair<int, int> keep = lower ? std::make_pair(lo, mid) : std::make_pair(mid, hi);
      const std::pair<int, int> send = lower ? std::make_pair(mid, hi) : std::make_pair(lo, mid);
      next[i] = keep;
      // partner i^d keeps exactly the half that i sends
      add_xfer(st, i, i ^ d, b[send.first], b[send.second], k == 1 ? RAW : PART, k == 1 ? RAW : PART,
               k == K ? RES : PART, k == K);
    }
    rng = next;
    p->steps.push_back(st);
  }
  for (int k = K; k >= 1; --k) {
    const int d = 1 << (k - 1);
    Step st{OP_COPY, {}};
    for (int i = 0; i < N; ++i) add_xfer(st, i, i ^ d, b[rng[i].first], b[rng[i].second], RES, RES, RES, false);
    std::vector<std::pair<int, int>> next(rng);
    for (int i = 0; i < N; ++i)
      next[i] = {std::min(rng[i].first, rng[i ^ d].first), std::max(rng[i].second, rng[i ^ d].second)};
    rng = next;
    p->steps.push_back(st);
  }
}

// Hierarchical all-reduce over M = N/G groups of G consecutive ranks (primer
// §4.4, Fig. 4.8 and Animation 4.3; AI Infra Book ch. 7, §7.2.1):
// (1) ring reduce-scatter inside each group, local rank l sending slice
//     (l - 1 - s) mod G, so that local rank k owns slice k;
// (2) for each slice k, a ring all-reduce among local rank k of every group,
//     over slice k cut into M sub-chunks;
// (3) ring all-gather inside each group, local rank l sending slice (l - s).
void build_hier(ar_plan_t* p) {
  const int N = p->desc.n_ranks, G = p->desc.group_size, M = N / G;
  const int64_t L = int64_t(p->desc.count);
  const auto sb = cuts(0, L, G);
  for (int s = 0; s <= G - 2; ++s) {  // phase 1
    Step st{OP_ADD, {}};
    const bool fin = (M == 1) && s == G - 2;
    for (int g = 0; g < M; ++g)
      for (int l = 0; l < G; ++l) {
        const int c = int(imod(l - 1 - s, G));
        add_xfer(st, g * G + l, g * G + (l + 1) % G, sb[c], sb[c + 1], s == 0 ? RAW : PART, RAW,
                 fin ? RES : PART, fin);
      }
    p->steps.push_back(st);
  }
  if (M > 1) {  // phase 2
    const Space own = G > 1 ? PART : RAW;
    for (int s = 0; s <= M - 2; ++s) {
      Step st{OP_ADD, {}};
      const bool fin = s == M - 2;
      for (int k = 0; k < G; ++k) {
        const auto sub = cuts(sb[k], sb[k + 1], M);
        for (int m = 0; m < M; ++m) {
          const int j = int(imod(m - s, M));
          add_xfer(st, m * G + k, ((m + 1) % M) * G + k, sub[j], sub[j + 1], s == 0 ? own : PART, own,
                   fin ? RES : PART, fin);
        }
      }
      p->steps.push_back(st);
    }
    for (int s = 0; s <= M - 2; ++s) {
      Step st{OP_COPY, {}};
      for (int k = 0; k < G; ++k) {
        const auto sub = cuts(sb[k], sb[k + 1], M);
        for (int m = 0; m < M; ++m) {
          const int j = int(imod(m + 1 - s, M));
          add_xfer(st, m * G + k, ((m + 1) % M) * G + k, sub[j], sub[j + 1], RES, RES, RES, false);
        }
      }
      p->steps.push_back(st);
    }
  }
  for (int s = 0; s <= G - 2; ++s) {  // phase 3
    Step st{OP_COPY, {}};
    for (int g = 0; g < M; ++g)
      for (int l = 0; l < G; ++l) {
        const int c = int(imod(l - s, G));
        add_xfer(st, g * G + l, g * G + (l + 1) % G, sb[c], sb[c + 1], RES, RES, RES, false);
      }
    p->steps.push_back(st);
  }
}

// Recursive doubling (primer §4.3, "Trees: latency-optimal, bandwidth-poor",
// Fig. 4.5): log2 N steps; in step k ranks i and i xor 2^(k-1) exchange their
// whole buffers and both add, so every rank holds the full sum at the end.
// One transfer per pair (from its lower rank) with `pair` set: the thread
// that adds an element writes the sum to both partners.
void build_recdoubling(ar_plan_t* p) {
  const int N = p->desc.n_ranks;
  const int64_t L = int64_t(p->desc.count);
  int K = 0;
  while ((1 << K) < N) ++K;
  for (int k = 1; k <= K; ++k) {
    const int d = 1 << (k - 1);
    Step st{OP_ADD, {}};
    const Space in = k == 1 ? RAW : PART;
    for (int i = 0; i < N; ++i) {
      if (i & d || L == 0) continue;
      Transfer t = make_xfer(i, i ^ d, 0, L, in, in, k == K ? RES : PART, k == K);
      t.pair = 1;
      st.xfers.push_back(t);
    }
    p->steps.push_back(st);
  }
}

// The two trees of the double binary tree (primer §4.3, Fig. 4.6). Tree 1:
// ranks 1..N-1 as the in-order binary tree -- rank r with lowest set bit
// b >= 2 has children r - b/2 and r + b/2, the right offset halved until the
// child is a rank below N -- whose top (the largest power of two below N)
// hangs under the root, rank 0; odd ranks are leaves. Tree 2 mirrors it:
// rank r becomes N-1-r. Children are kept in ascending rank order.
struct Tree {
  std::vector<int> parent, depth;
  std::vector<std::vector<int>> children;
};

std::vector<Tree> double_binary_trees(int N) {
  Tree t1;
  t1.parent.assign(N, -1);
  t1.children.assign(N, {});
  auto link = [&](int a, int c) {
    t1.parent[c] = a;
    t1.children[a].push_back(c);
  };
  if (N > 1) {
    int top = 1;
    while (top * 2 <= N - 1) top *= 2;
    link(0, top);
    for (int r = 1; r < N; ++r) {
      const int b = r & -r;
      if (b < 2) continue;
      link(r, r - b / 2);
      int off = b / 2;
      while (off >= 1 && r + off >= N) off /= 2;
      if (off >= 1) link(r, r + off);
    }
  }
  Tree t2;
  t2.parent.assign(N, -1);
  t2.children.assign(N, {});
  for (int r = 0; r < N; ++r) {
    const int m = N - 1 - r;
    if (t1.parent[r] >= 0) t2.parent[m] = N - 1 - t1.parent[r];
    for (int c : t1.children[r]) t2.children[m].push_back(N - 1 - c);
  }
  std::vector<Tree> trees = {t1, t2};
  for (Tree& t : trees) {
    for (auto& c : t.children) std::sort(c.begin(), c.end());
    t.depth.assign(N, 0);
    for (int r = 0; r < N; ++r)
      for (int q = r; t.parent[q] >= 0; q = t.parent[q]) ++t.depth[r];
  }
  return trees;
}

// All-reduce over the double binary tree: tree t carries half t of the
// buffer. Reduce, level by level from the deepest inner nodes up (both trees
// in the same steps: the mirror has the same levels): an inner node folds
// (own + first child) + second child into its partial sum, the root's sum
// is final (scaled and rounded once). Broadcast, from the root down: each
// parent's result overwrites its children's copies.
void build_dbtree(ar_plan_t* p) {
  const int N = p->desc.n_ranks;
  const int64_t L = int64_t(p->desc.count);
  const auto trees = double_binary_trees(N);
  const auto half = cuts(0, L, 2);
  int top = 0;
  for (const Tree& t : trees)
    for (int r = 0; r < N; ++r) top = std::max(top, t.depth[r]);
  for (int level = top - 1; level >= 0; --level) {
    Step st{OP_ADD, {}};
    for (int ti = 0; ti < 2; ++ti) {
      const Tree& t = trees[size_t(ti)];
      for (int r = 0; r < N; ++r) {
        const auto& ch = t.children[size_t(r)];
        if (t.depth[size_t(r)] != level || ch.empty() || half[ti + 1] <= half[ti]) continue;
        auto space = [&](int c) { return t.children[size_t(c)].empty() ? RAW : PART; };
        const bool root = t.parent[size_t(r)] < 0;
        Transfer x = make_xfer(ch[0], r, half[ti], half[ti + 1], space(ch[0]), RAW, root ? RES : PART, root);
        if (ch.size() > 1) {
          x.src2 = int16_t(ch[1]);
          x.x2s = space(ch[1]);
        }
        st.xfers.push_back(x);
      }
    }
    p->steps.push_back(st);
  }
  for (int level = 0; level < top; ++level) {
    Step st{OP_COPY, {}};
    for (int ti = 0; ti < 2; ++ti) {
      const Tree& t = trees[size_t(ti)];
      for (int r = 0; r < N; ++r)
        if (t.depth[size_t(r)] == level)
          for (int c : t.children[size_t(r)]) add_xfer(st, r, c, half[ti], half[ti + 1], RES, RES, RES, false);
    }
    p->steps.push_back(st);
  }
}

// Dimension-ordered all-reduce on an X x Y x Z torus (Scaling ML Systems,
// "Collective communication", torus section): rank (x, y, z) is
// x + X*(y + Y*z); dimension by dimension every line of ranks along it runs
// the ring all-reduce (ring rules as in build_ring, over the whole buffer cut
// into D chunks). Between dimensions the lines' sums stay fp32 partials; the
// last dimension's owners scale and round once.
void build_torus(ar_plan_t* p) {
  const int N = p->desc.n_ranks;
  const int64_t L = int64_t(p->desc.count);
  int dims[3];
  for (int k = 0; k < 3; ++k) dims[k] = std::max(p->desc.torus_dims[k], 1);
  const int stride[3] = {1, dims[0], dims[0] * dims[1]};
  int last = -1;
  for (int k = 0; k < 3; ++k)
    if (dims[k] > 1) last = k;
  bool first = true;
  for (int k = 0; k < 3; ++k) {
    const int D = dims[k];
    if (D == 1) continue;
    const auto b = cuts(0, L, D);
    std::vector<int> heads;  // first rank of every line along dimension k
    for (int r = 0; r < N; ++r)
      if ((r / stride[k]) % D == 0) heads.push_back(r);
    const bool fin_dim = k == last;
    for (int s = 0; s <= D - 2; ++s) {
      Step st{OP_ADD, {}};
      const bool fin = fin_dim && s == D - 2;
      for (int h : heads)
        for (int q = 0; q < D; ++q) {
          const int c = int(imod(q - s, D));
          const Space xs = first ? (s == 0 ? RAW : PART) : PART;
          add_xfer(st, h + q * stride[k], h + ((q + 1) % D) * stride[k], b[c], b[c + 1], xs, first ? RAW : PART,
                   fin ? RES : PART, fin);
        }
      p->steps.push_back(st);
    }
    const Space sp = fin_dim ? RES : PART;
    for (int s = 0; s <= D - 2; ++s) {
      Step st{OP_COPY, {}};
      for (int h : heads)
        for (int q = 0; q < D; ++q) {
          const int c = int(imod(q + 1 - s, D));
          add_xfer(st, h + q * stride[k], h + ((q + 1) % D) * stride[k], b[c], b[c + 1], sp, sp, sp, false);
        }
      p->steps.push_back(st);
    }
    first = false;
  }
}

size_t space_bytes(Space s, ar_dtype d) { return s == PART ? 4 : esize(d); }

// Every point-to-point send a transfer stands for: (src, dst, bytes per
// element). An exchange is two sends; a second source is one more.
template <class F>
void for_each_send(const Step& s, const Transfer& t, ar_dtype dt, F&& f) {
  f(int(t.src), int(t.dst), space_bytes(Space(t.xs), dt));
  if (s.op == OP_ADD && t.src2 >= 0) f(int(t.src2), int(t.dst), space_bytes(Space(t.x2s), dt));
  if (s.op == OP_ADD && t.pair) f(int(t.dst), int(t.src), space_bytes(Space(t.ys), dt));
}

int launches_of(const Step& s) { return int((s.xfers.size() + kMaxXfers - 1) / kMaxXfers); }

void compute_stats(ar_plan_t* p) {
  const ar_desc& d = p->desc;
  const int N = d.n_ranks;
  const int64_t L = int64_t(d.count);
  ar_stats& st = p->stats;
  st = ar_stats{};
  p->ws_stride = rup(std::max<int64_t>(L, 1), 64);
  if (d.algo == AR_FUSED) {
    const size_t es = esize(d.dtype), NL = size_t(N) * size_t(L);
    st.steps = N > 1 ? 1 : 0;
    st.launches = (L > 0 && N > 1) ? 1 : 0;
    if (d.collective == AR_ALLREDUCE) {  // every rank reads its buffer once and writes the sum once
      st.bytes_sent_per_rank = N > 1 ? size_t(L) * es : 0;
      st.hbm_bytes = N > 1 ? 2 * NL * es : 0;
    } else if (d.collective == AR_REDUCE_SCATTER) {  // N*S read, each chunk written once
      st.bytes_sent_per_rank = N > 1 ? size_t(L) * es : 0;
      st.hbm_bytes = N > 1 ? (NL + size_t(L)) * es : 0;
    } else {  // each chunk read once, written to every rank
      st.bytes_sent_per_rank = N > 1 ? ((size_t(L) + N - 1) / N) * es : 0;
      st.hbm_bytes = N > 1 ? (size_t(L) + NL) * es : 0;
    }
    st.workspace_bytes = 0;
    return;
  }
  st.steps = int(p->steps.size());
  std::vector<size_t> sent(N, 0);
  for (const Step& s : p->steps) {
    st.launches += launches_of(s);
    for (const Transfer& t : s.xfers) {
      const size_t len = size_t(t.hi - t.lo);
      for_each_send(s, t, d.dtype, [&](int src, int, size_t eb) { sent[size_t(src)] += len * eb; });
      // every operand read once and every destination written once
      size_t b = space_bytes(Space(t.xs), d.dtype) + space_bytes(Space(t.ds), d.dtype);
      if (s.op == OP_ADD) {
        b += space_bytes(Space(t.ys), d.dtype);
        if (t.src2 >= 0) b += space_bytes(Space(t.x2s), d.dtype);
        if (t.pair) b += space_bytes(Space(t.ds), d.dtype);
      }
      st.hbm_bytes += len * b;
    }
  }
  st.bytes_sent_per_rank = N > 0 ? *std::max_element(sent.begin(), sent.end()) : 0;
  const bool uses_ws = d.dtype == AR_BF16 && N > 1 && d.collective != AR_ALLGATHER;
  st.workspace_bytes = uses_ws ? size_t(N) * size_t(p->ws_stride) * 4 : 0;
  // Tiny steps: the whole schedule in one CTA when its table fits (room kept
  // for the all-gather's first copy of every rank's own chunk, L elements).
  int64_t n_x = 0, step_elems = L;
  for (const Step& s : p->steps) {
    n_x += int64_t(s.xfers.size());
    int64_t e = 0;
    for (const Transfer& t : s.xfers) e += t.hi - t.lo;
    step_elems = std::max(step_elems, e);
  }
  p->small = N > 1 && L > 0 && step_elems <= kSmallStepElems && n_x + N <= kMaxSmallXfers &&
             int64_t(p->steps.size()) + 1 <= kMaxSmallSteps;
  {  // on chip: the data fit, rows are whole 4-byte words, and the pieces fit the table
    int64_t pieces = 0;
    for (const Step& s : p->steps)
      for (const Transfer& t : s.xfers) pieces += (t.hi - t.lo + kSmallPiece - 1) / kSmallPiece;
    pieces += N + L / kSmallPiece;  // the all-gather's own-chunk copies, at most
    p->small_smem = p->small && small_smem_data_bytes(N, L) <= kSmallSmemDataBytes &&
                    (L * int64_t(esize(d.dtype))) % 4 == 0 && pieces <= kMaxSmallXfers;
  }
  if (p->small) st.launches = 1;
}

ar_status check_ptr(const void* ptr) {
  if (ptr == nullptr) return AR_EINVAL;
  if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return AR_EINVAL;
  return AR_OK;
}

// Every [start, start + bytes) must be disjoint from the others.
bool disjoint(std::vector<std::pair<uintptr_t, uintptr_t>> iv) {
  std::sort(iv.begin(), iv.end());
  for (size_t i = 1; i < iv.size(); ++i)
    if (iv[i].first < iv[i - 1].second) return false;
  return true;
}

ar_status check_buffers(const ar_plan_t* p, void* const* bufs, void* const* outs, void* workspace) {
  if (bufs == nullptr) return AR_EINVAL;
  const int N = p->desc.n_ranks;
  const size_t bytes = p->desc.count * esize(p->desc.dtype);
  std::vector<std::pair<uintptr_t, uintptr_t>> iv;
  for (int r = 0; r < N; ++r) {
    if (check_ptr(bufs[r]) != AR_OK) return AR_EINVAL;
    iv.push_back({uintptr_t(bufs[r]), uintptr_t(bufs[r]) + bytes});
    if (outs != nullptr) {
      if (check_ptr(outs[r]) != AR_OK) return AR_EINVAL;
      if (outs[r] != bufs[r]) iv.push_back({uintptr_t(outs[r]), uintptr_t(outs[r]) + bytes});
    }
  }
  if (p->stats.workspace_bytes > 0) {
    if (check_ptr(workspace) != AR_OK) return AR_EINVAL;
    iv.push_back({uintptr_t(workspace), uintptr_t(workspace) + p->stats.workspace_bytes});
  }
  if (bytes > 0 && !disjoint(iv)) return AR_EINVAL;
  return AR_OK;
}

ar_status from_cuda(cudaError_t e) { return e == cudaSuccess ? AR_OK : AR_ECUDA; }

// Before an executing call enqueues anything: publish the current device's
// host-visible status word (once per device) and refuse with AR_ETIMEOUT
// while a bounded device-side wait that ran out is still recorded in it
// (sticky until ar_device_status(1) clears it). Records the device on `p`.
ar_status status_guard(const ar_plan_t* p, int* device = nullptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return AR_ECUDA;
  volatile unsigned int* word = nullptr;
  if (host_status_word(dev, &word) != cudaSuccess) return AR_ECUDA;
  if (p != nullptr) p->last_device.v.store(dev, std::memory_order_relaxed);
  if (device != nullptr) *device = dev;
  return *word != 0 ? AR_ETIMEOUT : AR_OK;
}

// Segment count and tiles per segment of a fused launch over [e_lo, e_hi),
// for tiles of `tile` elements whose segment bodies start and end on
// multiples of W elements (the kernel's vector).
void fused_tiling(const ar_desc& d, FusedParams& fp, int64_t tile, int64_t W) {
  const int N = d.n_ranks;
  const int64_t L = int64_t(d.count);
  std::vector<std::pair<int64_t, int64_t>> segs;
  if (d.order == AR_ORDER_RING || d.collective != AR_ALLREDUCE) {
    const auto b = cuts(0, L, N);
    for (int c = 0; c < N; ++c) segs.push_back({b[c], b[c + 1]});
  } else if (d.order == AR_ORDER_HIER) {
    const int G = d.group_size, M = N / G;
    const auto sb = cuts(0, L, G);
    for (int k = 0; k < G; ++k) {
      const auto sub = cuts(sb[k], sb[k + 1], M);
      for (int j = 0; j < M; ++j) segs.push_back({sub[j], sub[j + 1]});
    }
  } else {
    segs.push_back({0, L});
  }
  int64_t tps = 1;
  for (auto& s : segs) {
    const int64_t lo = std::max(s.first, fp.e_lo), hi = std::min(s.second, fp.e_hi);
    if (hi <= lo) continue;
    const int64_t body = std::max<int64_t>(rdown(hi, W) - rup(lo, W), 0);
    tps = std::max(tps, (body + tile - 1) / tile);
  }
  fp.n_seg = int(segs.size());
  fp.tiles_per_seg = tps;
}

// `host_memory`: the buffers are pinned host memory read and written over the
// host link; only the register pipeline, whose plain loads and stores are
// known to work there, runs on them (the bulk-copy kernels are kept to device
// memory).
ar_status execute_fused(const ar_plan_t* p, void* const* bufs, void* const* outs, int64_t e_lo,
                        int64_t e_hi, cudaStream_t stream, bool host_memory = false) {
  const ar_desc& d = p->desc;
  FusedParams fp;
  std::memset(&fp, 0, sizeof(fp));
  for (int r = 0; r < d.n_ranks; ++r) {
    fp.in[r] = bufs[r];
    fp.out[r] = outs ? outs[r] : bufs[r];
  }
  fp.n = d.n_ranks;
  fp.collective = d.collective;
  fp.order = d.n_ranks == 1 && d.collective == AR_ALLREDUCE ? AR_ORDER_RANK : d.order;
  fp.g = d.order == AR_ORDER_HIER ? d.group_size : d.n_ranks;
  fp.m = d.order == AR_ORDER_HIER ? d.n_ranks / d.group_size : 1;
  fp.count = int64_t(d.count);
  fp.e_lo = e_lo;
  fp.e_hi = e_hi;
  fp.scale = d.collective == AR_ALLGATHER ? 1.0f : d.scale;  // an all-gather only copies
  int stages = 0, tile_bytes = 0;
  // the all-gather's bulk copies: faster from 96 MiB per rank (ar.h, AR_KERNEL_AUTO)
  const bool ag_bulk = d.kernel == AR_KERNEL_BULK ||
                       (d.kernel == AR_KERNEL_AUTO && d.count * esize(d.dtype) >= (size_t(96) << 20));
  if (!host_memory && ag_bulk && d.collective == AR_ALLGATHER && d.n_ranks > 1) {
    fused_tiling(d, fp, allgather_bulk_tile_elems(d.dtype), d.dtype == AR_BF16 ? 8 : 4);
    return from_cuda(launch_allgather_bulk(fp, d.dtype, d.sm_budget, stream));
  }
  if (!host_memory && d.kernel == AR_KERNEL_BULK && tma_shape(d.n_ranks, stages, tile_bytes)) {  // checked at plan time
    fused_tiling(d, fp, tile_bytes / int64_t(esize(d.dtype)), d.dtype == AR_BF16 ? 8 : 4);
    return from_cuda(launch_fused_tma(fp, d.dtype, stages, tile_bytes, d.sm_budget, stream));
  }
  fused_tiling(d, fp, fused_tile_elems(d.dtype, d.n_ranks, d.order, d.collective, budgeted(d.sm_budget)),
               fused_vec_elems(d.dtype, false));
  return from_cuda(launch_fused(fp, d.dtype, d.sm_budget, stream));
}

// `keep` (a plan that runs in one CTA only): fill *keep with the launch's
// parameters and *keep_smem with its kernel instead of launching (ar_bind).
ar_status execute_steps(const ar_plan_t* p, void* const* bufs, void* const* outs, void* workspace,
                        cudaStream_t stream, SmallParams* keep = nullptr, bool* keep_smem = nullptr) {
  const ar_desc& d = p->desc;
  const int N = d.n_ranks;
  static thread_local StepParams sp;  // ~3 KB, reused between calls
  std::memset(&sp, 0, sizeof(sp));
  for (int r = 0; r < N; ++r) {
    sp.raw[r] = bufs[r];
    sp.res[r] = outs ? outs[r] : bufs[r];
  }
  sp.ws = static_cast<float*>(workspace);
  sp.ws_stride = p->ws_stride;
  sp.scale = d.scale;
  sp.interleave = d.algo == AR_DBTREE ? 1 : 0;  // see the tile order in step.cu
  // 256-bit accesses when every base pointer is 32-byte aligned (see step.cu)
  bool v8 = workspace == nullptr || reinterpret_cast<uintptr_t>(workspace) % 32 == 0;
  for (int r = 0; r < N; ++r) {
    v8 = v8 && reinterpret_cast<uintptr_t>(bufs[r]) % 32 == 0;
    if (outs != nullptr) v8 = v8 && reinterpret_cast<uintptr_t>(outs[r]) % 32 == 0;
  }
  if (N == 1) {
    const bool in_place = outs == nullptr || outs[0] == bufs[0];
    const float scale = d.collective == AR_ALLGATHER ? 1.0f : d.scale;
    if (in_place && scale == 1.0f) return AR_OK;
    sp.scale = scale;
    sp.n_xfer = 1;
    sp.x[0] = make_xfer(0, 0, 0, int64_t(d.count), RAW, RAW, RES, true);
    sp.tile_start[0] = 0;
    const int64_t body = std::max<int64_t>(rdown(d.count, kStepVec), 0);
    sp.tile_start[1] = int32_t(std::max<int64_t>(1, (body + kStepTile - 1) / kStepTile));
    return from_cuda(launch_step(sp, d.dtype, OP_FINISH, sp.tile_start[1], false, d.sm_budget, v8, stream));
  }
  // out of place all-gather: every rank's own chunk is copied to its output
  // (the ring delivers only the other N-1 chunks): first, in a one-CTA plan;
  // by the first ring step otherwise (below)
  Step own{OP_COPY, {}};
  if (d.collective == AR_ALLGATHER && outs != nullptr) {
    const auto b = cuts(0, int64_t(d.count), N);
    for (int r = 0; r < N; ++r)
      if (outs[r] != bufs[r]) add_xfer(own, r, r, b[r], b[r + 1], RAW, RES, RES, false);
  }
  if (p->small) {  // the whole schedule in one CTA (step.cu)
    static thread_local SmallParams q;  // ~28 KB, reused between calls
    std::memset(&q, 0, sizeof(q));
    std::memcpy(q.raw, sp.raw, sizeof(q.raw));
    std::memcpy(q.res, sp.res, sizeof(q.res));
    q.ws = sp.ws;
    q.ws_stride = sp.ws_stride;
    q.scale = sp.scale;
    int nx = 0, ns = 0;
    auto add = [&](const Step& st) {
      q.step_start[ns] = nx;
      q.step_op[ns] = uint8_t(st.op);
      int32_t flat = 0;
      for (const Transfer& t : st.xfers) {
        SmallXfer& y = q.x[nx++];
        y.src = t.src;
        y.dst = t.dst;
        y.src2 = t.src2;
        y.xs = t.xs;
        y.ys = t.ys;
        y.ds = t.ds;
        y.x2s = t.x2s;
        y.fin = t.fin;
        y.pair = t.pair;
        y.lo = int32_t(t.lo);
        y.len = int32_t(t.hi - t.lo);
        y.flat = flat;
        flat += y.len;
      }
      q.step_elems[ns] = flat;
      ++ns;
    };
    // on chip: rows copied as words, so every buffer must be 4-byte aligned
    bool smem = p->small_smem, vec16 = (int64_t(d.count) * int64_t(esize(d.dtype))) % 16 == 0;
    for (int r = 0; r < N; ++r) {
      const uintptr_t a = reinterpret_cast<uintptr_t>(q.raw[r]), b = reinterpret_cast<uintptr_t>(q.res[r]);
      smem = smem && a % 4 == 0 && b % 4 == 0;
      vec16 = vec16 && a % 16 == 0 && b % 16 == 0;
    }
    if (smem) {  // the same steps, their transfers cut into pieces of one warp
      // The kernel's shared-memory layout (step.cu, small_steps_smem_kernel):
      // pieces, then (bf16) the fp32 partials, the inputs, the outputs.
      const int64_t L = int64_t(d.count), es = int64_t(esize(d.dtype));
      const bool bf = d.dtype == AR_BF16;
      int64_t n_pieces = 0;
      auto count_pieces = [&](const Step& st) {
        for (const Transfer& t : st.xfers) n_pieces += (t.hi - t.lo + kSmallPiece - 1) / kSmallPiece;
      };
      if (!own.xfers.empty()) count_pieces(own);
      for (const Step& st : p->steps) count_pieces(st);
      const int64_t tab = (n_pieces * int64_t(sizeof(SmemPiece)) + 15) / 16 * 16;
      const int64_t part0 = tab, raw0 = tab + (bf ? 4 * N * L : 0), res0 = raw0 + N * L * es;
      // (byte offset of element 0 of the operand, fp32?)
      auto where = [&](int space, int rank) -> std::pair<int64_t, bool> {
        const bool in_place = q.res[rank] == q.raw[rank];
        const int64_t in = raw0 + rank * L * es, out = in_place ? in : res0 + rank * L * es;
        if (space == RAW) return {in, !bf};
        if (space == RES) return {out, !bf};
        if (bf) return {part0 + rank * L * 4, true};
        return {out, true};
      };
      int widest = 1;
      auto add_pieces = [&](const Step& st) {
        q.step_start[ns] = nx;
        q.step_op[ns] = uint8_t(st.op);
        const int first = nx;
        for (const Transfer& t : st.xfers)
          for (int64_t lo = t.lo; lo < t.hi; lo += kSmallPiece) {
            SmemPiece& y = q.px[nx++];
            std::memset(&y, 0, sizeof(y));
            const auto X = where(t.xs, t.src), Y = where(t.ys, t.dst), D = where(t.ds, t.dst);
            y.x = uint32_t(X.first + lo * (X.second ? 4 : 2));
            y.y = uint32_t(Y.first + lo * (Y.second ? 4 : 2));
            y.d = uint32_t(D.first + lo * (D.second ? 4 : 2));
            y.flags = uint8_t((X.second ? kPieceX32 : 0) | (Y.second ? kPieceY32 : 0) | (D.second ? kPieceD32 : 0) |
                              (t.fin ? kPieceFin : 0));
            if (t.src2 >= 0) {
              const auto X2 = where(t.x2s, t.src2);
              y.x2 = uint32_t(X2.first + lo * (X2.second ? 4 : 2));
              y.flags |= uint8_t(kPieceTwo | (X2.second ? kPieceX2_32 : 0));
            }
            if (t.pair) {  // the partner's copy of the same space
              const auto D2 = where(t.ds, t.src);
              y.d2 = uint32_t(D2.first + lo * (D2.second ? 4 : 2));
              y.flags |= kPiecePair;
            }
            y.len = uint16_t(std::min<int64_t>(kSmallPiece, t.hi - lo));
          }
        widest = std::max(widest, nx - first);
        q.step_elems[ns] = 0;
        ++ns;
      };
      if (!own.xfers.empty()) add_pieces(own);
      for (const Step& st : p->steps) add_pieces(st);
      int threads = 128;  // at least 4 warps for the copies in and out
      while (threads < 32 * widest && threads < 1024) threads *= 2;
      q.threads = threads;
    } else {
      if (!own.xfers.empty()) add(own);
      for (const Step& st : p->steps) add(st);
    }
    q.step_start[ns] = nx;
    q.n_steps = ns;
    q.n_ranks = N;
    q.count = int32_t(d.count);
    q.in_place = 0;
    q.vec16 = vec16 ? 1 : 0;
    for (int r = 0; r < N; ++r)
      if (q.res[r] == q.raw[r]) q.in_place |= uint64_t(1) << r;
    if (keep != nullptr) {
      std::memcpy(keep, &q, sizeof(q));
      *keep_smem = smem;
      return AR_OK;
    }
    if (smem) return from_cuda(launch_small_steps_smem(q, d.dtype, stream));
    return from_cuda(launch_small_steps(q, d.dtype, stream));
  }
  // The own chunks ride on the all-gather's first step, which reads each of
  // them from its rank's input to send it: that step also writes it to the
  // sender's output (`pair`), saving a launch and a read of every chunk.
  std::vector<uint8_t> pair_first;
  if (!own.xfers.empty() && !p->steps.empty() && p->steps[0].op == OP_COPY) {
    const Step& first = p->steps[0];
    pair_first.assign(first.xfers.size(), 0);
    size_t matched = 0;
    for (const Transfer& o : own.xfers)
      for (size_t x = 0; x < first.xfers.size(); ++x) {
        const Transfer& t = first.xfers[x];
        if (t.src == o.src && t.lo == o.lo && t.hi == o.hi && t.xs == RAW && t.ds == RES && !pair_first[x]) {
          pair_first[x] = 1;
          ++matched;
          break;
        }
      }
    if (matched == own.xfers.size())
      own.xfers.clear();
    else
      pair_first.clear();
  }
  if (!own.xfers.empty()) {
    sp.n_xfer = int(own.xfers.size());
    int tiles = 0;
    for (int x = 0; x < sp.n_xfer; ++x) {
      const Transfer& t = own.xfers[size_t(x)];
      sp.x[x] = t;
      sp.tile_start[x] = tiles;
      const int64_t body = std::max<int64_t>(rdown(t.hi, kStepVec) - rup(t.lo, kStepVec), 0);
      tiles += int(std::max<int64_t>(1, (body + kStepTile - 1) / kStepTile));
    }
    sp.tile_start[sp.n_xfer] = tiles;
    const ar_status s = from_cuda(launch_step(sp, d.dtype, OP_COPY, tiles, true, d.sm_budget, v8, stream));
    if (s != AR_OK) return s;
  }
  for (const Step& st : p->steps) {
    // A bf16 copy step whose transfers all start and end on an even element
    // and move bf16 buffers (not the fp32 partials) runs as an fp32 copy of
    // element pairs over the same bytes: 32-byte vectors when the buffers
    // allow them, half the instructions per byte.
    bool pairs = d.dtype == AR_BF16 && st.op == OP_COPY;
    for (const Transfer& t : st.xfers)
      pairs = pairs && t.lo % 2 == 0 && t.hi % 2 == 0 && t.xs != PART && t.ds != PART;
    const int64_t div = pairs ? 2 : 1;
    // a step's transfers are independent (none writes what another reads), so
    // a step with more transfers than one launch holds runs as several
    for (size_t x0 = 0; x0 < st.xfers.size(); x0 += kMaxXfers) {
      sp.n_xfer = int(std::min<size_t>(kMaxXfers, st.xfers.size() - x0));
      int tiles = 0;
      for (int x = 0; x < sp.n_xfer; ++x) {
        const Transfer& t = st.xfers[x0 + size_t(x)];
        sp.x[x] = t;
        sp.x[x].lo = t.lo / div;
        sp.x[x].hi = t.hi / div;
        if (&st == &p->steps[0] && !pair_first.empty()) sp.x[x].pair = pair_first[x0 + size_t(x)];
        sp.tile_start[x] = tiles;
        const Transfer& u = sp.x[x];
        const int64_t body = std::max<int64_t>(rdown(u.hi, kStepVec) - rup(u.lo, kStepVec), 0);
        tiles += int(std::max<int64_t>(1, (body + kStepTile - 1) / kStepTile));
      }
      sp.tile_start[sp.n_xfer] = tiles;
      const ar_status s =
          from_cuda(launch_step(sp, pairs ? AR_F32 : d.dtype, st.op, tiles, true, d.sm_budget, v8, stream));
      if (s != AR_OK) return s;
    }
  }
  return AR_OK;
}

// Internal streams and events of ar_execute_host, one set per device.
struct HostPipe {
  int device = -1;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  std::vector<cudaEvent_t> ev;
};
std::mutex g_host_mu;
std::vector<HostPipe> g_pipes;

ar_status host_pipe(HostPipe** out, size_t n_events) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return AR_ECUDA;
  HostPipe* hp = nullptr;
  for (auto& x : g_pipes)
    if (x.device == dev) hp = &x;
  if (hp == nullptr) {
    g_pipes.push_back(HostPipe{});
    hp = &g_pipes.back();
    hp->device = dev;
    if (cudaStreamCreateWithFlags(&hp->h2d, cudaStreamNonBlocking) != cudaSuccess) return AR_ECUDA;
    if (cudaStreamCreateWithFlags(&hp->d2h, cudaStreamNonBlocking) != cudaSuccess) return AR_ECUDA;
  }
  while (hp->ev.size() < n_events) {
    cudaEvent_t e;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return AR_ECUDA;
    hp->ev.push_back(e);
  }
  *out = hp;
  return AR_OK;
}

}  // namespace

extern "C" {

ar_status ar_plan(const ar_desc* desc, ar_plan_t** out) {
  if (desc == nullptr || out == nullptr) return AR_EINVAL;
  *out = nullptr;
  const ar_desc& d = *desc;
  const int N = d.n_ranks;
  if (N < 1 || N > AR_MAX_RANKS) return AR_EINVAL;
  if (d.dtype != AR_F32 && d.dtype != AR_BF16) return AR_EINVAL;
  if (d.algo == AR_AUTO) {  // resolve under this GPU's own fabric, then plan the choice
    const ar_fabric dev = {AR_DEVICE_ALPHA_S, AR_DEVICE_BW, AR_DEVICE_BW, 0, 0, 1};
    ar_desc r = d;
    r.algo = AR_FUSED;
    int gs = 0;
    const ar_status s = ar_select(&d, &dev, &r.algo, &gs, nullptr);
    if (s != AR_OK) return s;
    if (r.algo == AR_HIER) r.group_size = gs;
    return ar_plan(&r, out);
  }
  if (d.algo < AR_RING || d.algo > AR_TORUS || d.algo == AR_AUTO) return AR_EINVAL;
  if (!std::isfinite(d.scale)) return AR_EINVAL;
  if (d.count > (size_t(1) << 40)) return AR_EINVAL;
  if (d.collective < AR_ALLREDUCE || d.collective > AR_ALLGATHER) return AR_EINVAL;
  if (d.sm_budget < 0) return AR_EINVAL;
  if (d.kernel < AR_KERNEL_AUTO || d.kernel > AR_KERNEL_BULK) return AR_EINVAL;
  if (d.kernel == AR_KERNEL_BULK && d.algo == AR_FUSED && N > 1) {
    int stages = 0, tile_bytes = 0;
    const bool ok = d.collective == AR_ALLGATHER || (d.collective == AR_ALLREDUCE && tma_shape(N, stages, tile_bytes));
    if (!ok) return AR_EUNSUPPORTED;
  }
  if (d.algo == AR_TORUS) {
    int prod = 1;
    for (int k = 0; k < 3; ++k) {
      if (d.torus_dims[k] < 0 || d.torus_dims[k] > AR_MAX_RANKS) return AR_EINVAL;
      prod *= std::max(d.torus_dims[k], 1);
    }
    if (prod != N) return AR_EINVAL;
  }
  if (d.collective != AR_ALLREDUCE) {
    if (d.algo != AR_RING && d.algo != AR_FUSED) return AR_EUNSUPPORTED;
    if (d.algo == AR_FUSED && d.order == AR_ORDER_HIER) return AR_EUNSUPPORTED;
  }
  if ((d.algo == AR_RABENSEIFNER || d.algo == AR_RECDOUBLING) && !is_pow2(N)) return AR_EINVAL;
  if (d.algo == AR_HIER && (d.group_size < 1 || N % d.group_size != 0)) return AR_EINVAL;
  if (d.algo == AR_FUSED) {
    if (d.order < AR_ORDER_RING || d.order > AR_ORDER_HIER) return AR_EINVAL;
    if (d.order == AR_ORDER_TREE && !is_pow2(N)) return AR_EINVAL;
    if (d.order == AR_ORDER_HIER && (d.group_size < 1 || N % d.group_size != 0)) return AR_EINVAL;
  }
  ar_plan_t* p = new (std::nothrow) ar_plan_t;
  if (p == nullptr) return AR_ENOMEM;
  try {
    p->desc = d;
    if (d.algo != AR_HIER && !(d.algo == AR_FUSED && d.order == AR_ORDER_HIER)) p->desc.group_size = 0;
    if (d.algo != AR_TORUS)
      for (int k = 0; k < 3; ++k) p->desc.torus_dims[k] = 0;
    if (N > 1 && d.collective == AR_REDUCE_SCATTER) build_ring_reduce_scatter(p);
    if (N > 1 && d.collective == AR_ALLGATHER) build_ring_allgather(p);
    if (N > 1 && d.collective == AR_ALLREDUCE) {
      if (d.algo == AR_RING) build_ring(p);
      if (d.algo == AR_RABENSEIFNER) build_rabenseifner(p);
      if (d.algo == AR_HIER) build_hier(p);
      if (d.algo == AR_RECDOUBLING) build_recdoubling(p);
      if (d.algo == AR_DBTREE) build_dbtree(p);
      if (d.algo == AR_TORUS) build_torus(p);
    }
    compute_stats(p);
  } catch (const std::bad_alloc&) {
    delete p;
    return AR_ENOMEM;
  }
  *out = p;
  return AR_OK;
}

ar_status ar_plan_stats(const ar_plan_t* plan, ar_stats* stats) {
  if (plan == nullptr || stats == nullptr) return AR_EINVAL;
  *stats = plan->stats;
  return AR_OK;
}

ar_status ar_plan_desc(const ar_plan_t* plan, ar_desc* desc) {
  if (plan == nullptr || desc == nullptr) return AR_EINVAL;
  *desc = plan->desc;
  return AR_OK;
}

void ar_plan_destroy(ar_plan_t* plan) { delete plan; }

ar_status ar_plan_transfers(const ar_plan_t* plan, int step, int* op, int* n_xfers, int64_t* xfers,
                            int max_xfers) {
  if (plan == nullptr || op == nullptr || n_xfers == nullptr) return AR_EINVAL;
  if (plan->desc.algo == AR_FUSED || step < 0 || step >= int(plan->steps.size())) return AR_EINVAL;
  const Step& st = plan->steps[size_t(step)];
  *op = st.op == OP_ADD ? 0 : 1;
  int n = 0;
  for (const Transfer& t : st.xfers)
    for_each_send(st, t, plan->desc.dtype, [&](int src, int dst, size_t) {
      if (xfers != nullptr && n < max_xfers) {
        xfers[4 * n + 0] = src;
        xfers[4 * n + 1] = dst;
        xfers[4 * n + 2] = t.lo;
        xfers[4 * n + 3] = t.hi;
      }
      ++n;
    });
  *n_xfers = n;
  return AR_OK;
}

ar_status ar_execute(const ar_plan_t* plan, void* const* bufs, void* const* outs, void* workspace,
                     void* stream) {
  if (plan == nullptr) return AR_EINVAL;
  const ar_status s = check_buffers(plan, bufs, outs, workspace);
  if (s != AR_OK) return s;
  if (plan->desc.count == 0) return AR_OK;
  const ar_status g = status_guard(plan);
  if (g != AR_OK) return g;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (plan->desc.algo == AR_FUSED)
    return execute_fused(plan, bufs, outs, 0, int64_t(plan->desc.count), st);
  return execute_steps(plan, bufs, outs, workspace, st);
}

}  // extern "C"

// A plan bound to its buffers. Step plans: the launches of one ar_execute
// recorded once into a CUDA graph (ar_bind) and replayed by ar_execute_bound.
// Single-pass plans are one kernel, which a direct launch starts sooner than
// a one-node graph (measured on GB300: 3.8 against 6.2 us per call back to
// back), so they keep the validated plan and buffers and launch directly.
// So do step plans that run whole in one CTA: their launch parameters are
// built once, here, and launched as they are on every call.
struct ar_bound {
  int device = -1;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  struct ar_plan plan;          // fused: a copy of the plan (its descriptor and stats)
  std::vector<void*> bufs, outs;
  bool direct = false;
  std::unique_ptr<ar::SmallParams> small;  // one-CTA step plan: its launch parameters
  bool small_smem = false;
  ar_dtype dtype = AR_F32;
};

namespace {

void release(ar_bound* b) {
  if (b == nullptr) return;
  if (b->exec != nullptr) cudaGraphExecDestroy(b->exec);
  if (b->graph != nullptr) cudaGraphDestroy(b->graph);
  delete b;
}

}  // namespace

extern "C" {

ar_status ar_bind(const ar_plan_t* plan, void* const* bufs, void* const* outs, void* workspace, ar_bound_t** out) {
  if (plan == nullptr || out == nullptr) return AR_EINVAL;
  *out = nullptr;
  const ar_status chk = check_buffers(plan, bufs, outs, workspace);
  if (chk != AR_OK) return chk;
  ar_bound* b = new (std::nothrow) ar_bound;
  if (b == nullptr) return AR_ENOMEM;
  if (plan->desc.count == 0) {  // nothing to launch: no graph, no CUDA call
    *out = b;
    return AR_OK;
  }
  const ar_status g = status_guard(plan, &b->device);  // also publishes the word before any capture
  if (g != AR_OK) {
    release(b);
    return g;
  }
  if (plan->desc.algo == AR_FUSED) {
    b->plan = *plan;
    const int N = plan->desc.n_ranks;
    b->bufs.assign(bufs, bufs + N);
    if (outs != nullptr) b->outs.assign(outs, outs + N);
    b->direct = true;
    *out = b;
    return AR_OK;
  }
  if (plan->small) {  // one CTA: the parameters once, a direct launch per call
    b->small.reset(new (std::nothrow) ar::SmallParams);
    if (!b->small) {
      release(b);
      return AR_ENOMEM;
    }
    b->dtype = plan->desc.dtype;
    const ar_status s = execute_steps(plan, bufs, outs, workspace, nullptr, b->small.get(), &b->small_smem);
    if (s != AR_OK) {
      release(b);
      return s;
    }
    *out = b;
    return AR_OK;
  }
  // Record on a private stream. Relaxed mode: the launchers' first-use
  // occupancy queries are allowed while capturing.
  cudaStream_t cap = nullptr;
  if (cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking) != cudaSuccess) {
    release(b);
    return AR_ECUDA;
  }
  ar_status s = AR_OK;
  if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    s = AR_ECUDA;
  } else {
    s = execute_steps(plan, bufs, outs, workspace, cap);
    const cudaError_t e = cudaStreamEndCapture(cap, &b->graph);  // ends the capture even after an error
    if (s == AR_OK && e != cudaSuccess) s = AR_ECUDA;
  }
  cudaStreamDestroy(cap);
  if (s == AR_OK && cudaGraphInstantiate(&b->exec, b->graph, 0) != cudaSuccess) s = AR_ECUDA;
  if (s != AR_OK) {
    release(b);
    return s;
  }
  *out = b;
  return AR_OK;
}

ar_status ar_execute_bound(const ar_bound_t* bound, void* stream) {
  if (bound == nullptr) return AR_EINVAL;
  if (bound->exec == nullptr && !bound->direct && !bound->small) return AR_OK;  // count == 0
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return AR_ECUDA;
  if (dev != bound->device) return AR_EINVAL;
  const volatile unsigned int* word = host_status_word_if_ready(dev);  // published by ar_bind
  if (word == nullptr) return AR_ECUDA;
  if (*word != 0) return AR_ETIMEOUT;
  if (bound->direct)
    return execute_fused(&bound->plan, bound->bufs.data(), bound->outs.empty() ? nullptr : bound->outs.data(), 0,
                         int64_t(bound->plan.desc.count), static_cast<cudaStream_t>(stream));
  if (bound->small)
    return from_cuda(bound->small_smem
                         ? launch_small_steps_smem(*bound->small, bound->dtype, static_cast<cudaStream_t>(stream))
                         : launch_small_steps(*bound->small, bound->dtype, static_cast<cudaStream_t>(stream)));
  return from_cuda(cudaGraphLaunch(bound->exec, static_cast<cudaStream_t>(stream)));
}

void ar_bound_destroy(ar_bound_t* bound) { release(bound); }

ar_status ar_execute_host(const ar_plan_t* plan, const void* const* host_in, void* const* host_out,
                          void* const* dev_bufs, void* workspace, void* stream) {
  if (plan == nullptr || host_in == nullptr || host_out == nullptr) return AR_EINVAL;
  const ar_status s = check_buffers(plan, dev_bufs, nullptr, workspace);
  if (s != AR_OK) return s;
  const int N = plan->desc.n_ranks;
  for (int r = 0; r < N; ++r)
    if (host_in[r] == nullptr || host_out[r] == nullptr) return AR_EINVAL;
  const int64_t L = int64_t(plan->desc.count);
  if (L == 0) return AR_OK;
  const ar_status g = status_guard(plan);
  if (g != AR_OK) return g;
  const size_t es = esize(plan->desc.dtype);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_host_mu);

  if (plan->desc.algo == AR_FUSED) {
    // Page-locked host memory on a unified-address system is directly
    // readable and writable by kernels: over NVLink-C2C the single pass then
    // reads host_in and writes host_out itself, with no staging copies.
    std::vector<void*> in_dev(N, nullptr), out_dev(N, nullptr);
    bool direct = true;
    for (int r = 0; r < N && direct; ++r) {
      cudaPointerAttributes a{}, b{};
      if (cudaPointerGetAttributes(&a, host_in[r]) != cudaSuccess ||
          cudaPointerGetAttributes(&b, host_out[r]) != cudaSuccess) {
        cudaGetLastError();  // pageable memory on some drivers reports an error: not direct
        direct = false;
        break;
      }
      direct = a.type == cudaMemoryTypeHost && b.type == cudaMemoryTypeHost && a.devicePointer != nullptr &&
               b.devicePointer != nullptr;
      in_dev[r] = a.devicePointer;
      out_dev[r] = b.devicePointer;
    }
    if (direct) {
      const ar_status e = check_buffers(plan, in_dev.data(), out_dev.data(), nullptr);
      if (e != AR_OK) return e;
      const ar_status x = execute_fused(plan, in_dev.data(), out_dev.data(), 0, L, st, true);
      if (x != AR_OK) return x;
      return from_cuda(cudaStreamSynchronize(st));
    }
  }

  if (plan->desc.algo != AR_FUSED) {  // the schedule spans the whole buffer: copy, run, copy
    for (int r = 0; r < N; ++r)
      if (cudaMemcpyAsync(dev_bufs[r], host_in[r], size_t(L) * es, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return AR_ECUDA;
    const ar_status e = ar_execute(plan, dev_bufs, nullptr, workspace, stream);
    if (e != AR_OK) return e;
    for (int r = 0; r < N; ++r)
      if (cudaMemcpyAsync(host_out[r], dev_bufs[r], size_t(L) * es, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return AR_ECUDA;
    return from_cuda(cudaStreamSynchronize(st));
  }

  // Fused: elements are independent, so the buffers are cut into slabs of
  // whole 16-byte vectors; slab k's host-to-device copies, its reduction and
  // its device-to-host copies run on three streams, overlapping the copies of
  // neighbouring slabs in both directions with the reduction.
  const int64_t target = std::max<int64_t>(int64_t(64) << 20, 0) / int64_t(es) / N;  // ~64 MiB per slab
  const int64_t slab = std::max<int64_t>(rup(std::min<int64_t>(target, L), 64), 64);
  const int64_t n_slabs = (L + slab - 1) / slab;
  HostPipe* hp = nullptr;
  ar_status e = host_pipe(&hp, size_t(2 * n_slabs + 1));
  if (e != AR_OK) return e;
  // copies must not start before earlier work on the caller's stream
  cudaEvent_t start = hp->ev[2 * n_slabs];
  if (cudaEventRecord(start, st) != cudaSuccess) return AR_ECUDA;
  if (cudaStreamWaitEvent(hp->h2d, start, 0) != cudaSuccess) return AR_ECUDA;
  for (int64_t k = 0; k < n_slabs; ++k) {
    const int64_t lo = k * slab, hi = std::min(L, lo + slab);
    for (int r = 0; r < N; ++r)
      if (cudaMemcpyAsync(static_cast<char*>(dev_bufs[r]) + lo * es,
                          static_cast<const char*>(host_in[r]) + lo * es, size_t(hi - lo) * es,
                          cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess)
        return AR_ECUDA;
    cudaEvent_t copied = hp->ev[2 * k], reduced = hp->ev[2 * k + 1];
    if (cudaEventRecord(copied, hp->h2d) != cudaSuccess) return AR_ECUDA;
    if (cudaStreamWaitEvent(st, copied, 0) != cudaSuccess) return AR_ECUDA;
    e = execute_fused(plan, dev_bufs, nullptr, lo, hi, st);
    if (e != AR_OK) return e;
    if (cudaEventRecord(reduced, st) != cudaSuccess) return AR_ECUDA;
    if (cudaStreamWaitEvent(hp->d2h, reduced, 0) != cudaSuccess) return AR_ECUDA;
    for (int r = 0; r < N; ++r)
      if (cudaMemcpyAsync(static_cast<char*>(host_out[r]) + lo * es,
                          static_cast<const char*>(dev_bufs[r]) + lo * es, size_t(hi - lo) * es,
                          cudaMemcpyDeviceToHost, hp->d2h) != cudaSuccess)
        return AR_ECUDA;
  }
  return from_cuda(cudaStreamSynchronize(hp->d2h));
}

// ---------------------------------------------------------------- cost model

static bool fabric_ok(const ar_fabric* f) {
  auto pos = [](double x) { return std::isfinite(x) && x > 0; };
  return f != nullptr && std::isfinite(f->alpha) && f->alpha >= 0 && pos(f->bw_local) &&
         (f->shared_memory || pos(f->bw_net)) && f->ranks_per_server >= 0;
}

ar_status ar_plan_predict(const ar_plan_t* plan, const ar_fabric* f, double* seconds) {
  if (plan == nullptr || seconds == nullptr || !fabric_ok(f)) return AR_EINVAL;
  const ar_desc& d = plan->desc;
  const ar_stats& st = plan->stats;
  const int N = d.n_ranks, rps = f->ranks_per_server;
  if (f->shared_memory) {  // one memory for all ranks: each launch, the in-CTA steps, then all its bytes
    const double per_step = plan->small_smem ? AR_DEVICE_CTA_STEP_S : AR_DEVICE_CTA_STEP_MEM_S;
    const double cta_steps = plan->small ? double(st.steps) * per_step : 0.0;
    *seconds = st.launches * f->alpha + cta_steps + double(st.hbm_bytes) / f->bw_local;
    return AR_OK;
  }
  if (d.algo == AR_FUSED) {
    if (!f->in_network) return AR_EUNSUPPORTED;
    const bool multi = rps > 0 && N > rps;
    // one round: a rank sends its whole buffer up (reduce-scatter, all-reduce)
    // or receives the whole result (all-gather, all-reduce)
    *seconds = N > 1 ? f->alpha + double(d.count) * esize(d.dtype) / (multi ? f->bw_net : f->bw_local) : 0.0;
    return AR_OK;
  }
  auto bw = [&](int a, int b) {
    return (rps == 0 || a / rps == b / rps) ? f->bw_local : f->bw_net;
  };
  double T = 0;
  for (const Step& s : plan->steps) {
    double worst = 0;
    for (const Transfer& t : s.xfers)
      for_each_send(s, t, d.dtype, [&](int src, int dst, size_t eb) {
        worst = std::max(worst, double(t.hi - t.lo) * double(eb) / bw(src, dst));
      });
    T += f->alpha + worst;
  }
  *seconds = T;
  return AR_OK;
}

ar_status ar_select(const ar_desc* desc, const ar_fabric* f, ar_algo* algo, int* group_size,
                    double* seconds) {
  if (desc == nullptr || algo == nullptr || !fabric_ok(f)) return AR_EINVAL;
  const int N = desc->n_ranks;
  // earlier candidates win ties: the single pass first (with N = 2 an
  // exchange moves the same bytes in the same one step)
  std::vector<std::pair<ar_algo, int>> cand;
  if (f->in_network || f->shared_memory) cand.push_back({AR_FUSED, 0});
  cand.push_back({AR_RING, 0});
  if (desc->collective == AR_ALLREDUCE) {
    if (is_pow2(N)) cand.push_back({AR_RABENSEIFNER, 0});
    if (is_pow2(N)) cand.push_back({AR_RECDOUBLING, 0});
    cand.push_back({AR_DBTREE, 0});
    const int G = f->ranks_per_server;
    if (G > 1 && G < N && N % G == 0) cand.push_back({AR_HIER, G});
  }
  bool found = false;
  double best = 0;
  ar_status last = AR_EINVAL;
  for (const auto& c : cand) {
    ar_desc d = *desc;
    d.algo = c.first;
    if (c.first == AR_HIER) d.group_size = c.second;
    if (c.first == AR_FUSED && d.order == AR_ORDER_HIER && d.collective != AR_ALLREDUCE) d.order = AR_ORDER_RING;
    ar_plan_t* p = nullptr;
    last = ar_plan(&d, &p);
    if (last != AR_OK) continue;
    double t = 0;
    last = ar_plan_predict(p, f, &t);
    const int gs = p->desc.group_size;
    ar_plan_destroy(p);
    if (last != AR_OK) continue;
    if (!found || t < best) {
      found = true;
      best = t;
      *algo = c.first;
      if (group_size) *group_size = gs;
    }
  }
  if (!found) return last;
  if (seconds) *seconds = best;
  return AR_OK;
}

// ---------------------------------------------------------------- buckets

ar_status ar_bucket_plan(const size_t* counts, int n_tensors, size_t elem_bytes, size_t cap_bytes,
                         int* bucket_of_tensor, int* n_buckets) {
  if (counts == nullptr || bucket_of_tensor == nullptr || n_buckets == nullptr) return AR_EINVAL;
  if (n_tensors < 1 || elem_bytes == 0) return AR_EINVAL;
  int b = 0;
  size_t cur = 0;
  bool open = false;
  for (int t = n_tensors - 1; t >= 0; --t) {  // backward produces the last tensor first
    const size_t bytes = counts[t] * elem_bytes;
    if (open && cur + bytes > cap_bytes) {
      ++b;
      cur = 0;
    }
    bucket_of_tensor[t] = b;
    cur += bytes;
    open = true;
  }
  *n_buckets = b + 1;
  return AR_OK;
}

namespace {

ar_status check_bucket_args(int n_ranks, const void* const* tensors, const size_t* counts, int n_tensors,
                            int t_begin, int t_end) {
  if (n_ranks < 1 || n_ranks > AR_MAX_RANKS) return AR_EINVAL;
  if (tensors == nullptr || counts == nullptr) return AR_EINVAL;
  if (n_tensors < 1 || t_begin < 0 || t_end > n_tensors || t_begin >= t_end) return AR_EINVAL;
  for (int t = t_begin; t < t_end; ++t)
    for (int r = 0; r < n_ranks; ++r)
      if (check_ptr(tensors[size_t(r) * n_tensors + t]) != AR_OK) return AR_EINVAL;
  return AR_OK;
}

// Packed offset of each tensor of bucket [t_begin, t_end): descending ids.
std::vector<int64_t> packed_offsets(const size_t* counts, int t_begin, int t_end) {
  std::vector<int64_t> off(t_end - t_begin);
  int64_t o = 0;
  for (int t = t_end - 1; t >= t_begin; --t) {
    off[t - t_begin] = o;
    o += int64_t(counts[t]);
  }
  return off;
}

ar_status run_pack(int n_ranks, const void* const* tensors, const size_t* counts, int n_tensors,
                   int t_begin, int t_end, ar_dtype dtype, void* const* bucket, float scale, bool unpack,
                   cudaStream_t stream) {
  const auto off = packed_offsets(counts, t_begin, t_end);
  const int max_group = std::min(AR_MAX_BUCKET_TENSORS, kMaxBucketPtrs / n_ranks);
  static thread_local PackParams pp;
  for (int g0 = t_end - 1; g0 >= t_begin; g0 -= max_group) {  // groups of tensors, packing order
    std::memset(&pp, 0, sizeof(pp));
    pp.n = n_ranks;
    pp.scale = scale;
    int nt = 0, tiles = 0;
    for (int t = g0; t >= t_begin && nt < max_group; --t, ++nt) {
      for (int r = 0; r < n_ranks; ++r) pp.tptr[nt * n_ranks + r] = const_cast<void*>(tensors[size_t(r) * n_tensors + t]);
      pp.off[nt] = off[t - t_begin];
      pp.cnt[nt] = int64_t(counts[t]);
      pp.tile_start[nt] = tiles;
      tiles += int((int64_t(counts[t]) + kPackTile - 1) / kPackTile);
    }
    pp.n_t = nt;
    pp.tile_start[nt] = tiles;
    for (int r = 0; r < n_ranks; ++r) pp.bucket[r] = bucket[r];
    if (launch_pack(pp, dtype, unpack, stream) != cudaSuccess) return AR_ECUDA;
  }
  return AR_OK;
}

}  // namespace

ar_status ar_bucket_pack(int n_ranks, const void* const* tensors, const size_t* counts, int n_tensors,
                         int t_begin, int t_end, ar_dtype in_dtype, void* const* bucket, void* stream) {
  ar_status s = check_bucket_args(n_ranks, tensors, counts, n_tensors, t_begin, t_end);
  if (s != AR_OK) return s;
  if (in_dtype != AR_F32 && in_dtype != AR_BF16) return AR_EINVAL;
  if (bucket == nullptr) return AR_EINVAL;
  for (int r = 0; r < n_ranks; ++r)
    if (check_ptr(bucket[r]) != AR_OK) return AR_EINVAL;
  return run_pack(n_ranks, tensors, counts, n_tensors, t_begin, t_end, in_dtype, bucket, 1.0f, false,
                  static_cast<cudaStream_t>(stream));
}

ar_status ar_bucket_unpack(int n_ranks, const void* const* bucket, float scale, ar_dtype out_dtype,
                           void* const* tensors, const size_t* counts, int n_tensors, int t_begin, int t_end,
                           void* stream) {
  ar_status s = check_bucket_args(n_ranks, tensors, counts, n_tensors, t_begin, t_end);
  if (s != AR_OK) return s;
  if (out_dtype != AR_F32 && out_dtype != AR_BF16) return AR_EINVAL;
  if (bucket == nullptr || !std::isfinite(scale)) return AR_EINVAL;
  for (int r = 0; r < n_ranks; ++r)
    if (check_ptr(bucket[r]) != AR_OK) return AR_EINVAL;
  return run_pack(n_ranks, tensors, counts, n_tensors, t_begin, t_end, out_dtype,
                  const_cast<void* const*>(bucket), scale, true, static_cast<cudaStream_t>(stream));
}

ar_status ar_bucket_allreduce(int n_ranks, void* const* tensors, const size_t* counts, int n_tensors,
                              int t_begin, int t_end, ar_dtype dtype, float scale, int sm_budget,
                              ar_kernel kernel, void* stream) {
  ar_status s = check_bucket_args(n_ranks, tensors, counts, n_tensors, t_begin, t_end);
  if (s != AR_OK) return s;
  if (dtype != AR_F32 && dtype != AR_BF16) return AR_EINVAL;
  if (!std::isfinite(scale) || sm_budget < 0) return AR_EINVAL;
  if (kernel < AR_KERNEL_AUTO || kernel > AR_KERNEL_BULK) return AR_EINVAL;
  const int N = n_ranks;
  const auto off = packed_offsets(counts, t_begin, t_end);
  int64_t Lb = 0;
  for (int t = t_begin; t < t_end; ++t) Lb += int64_t(counts[t]);
  if (Lb == 0) return AR_OK;
  const auto b = cuts(0, Lb, N);
  int stages = 0, tile_bytes = 0;
  const bool tma = kernel == AR_KERNEL_BULK;
  bool v8 = !tma && N > 4;  // 32-byte vectors when every tensor of the bucket is 32-byte aligned
  for (int t = t_begin; t < t_end && v8; ++t)
    for (int r = 0; r < N; ++r)
      if (reinterpret_cast<uintptr_t>(tensors[size_t(r) * n_tensors + t]) % 32 != 0) v8 = false;
  const int64_t W = tma ? (dtype == AR_BF16 ? 8 : 4) : fused_vec_elems(dtype, v8);  // the kernel's vector
  if (tma && !tma_shape(N, stages, tile_bytes)) return AR_EUNSUPPORTED;
  s = status_guard(nullptr);
  if (s != AR_OK) return s;
  const int64_t tile = tma ? tile_bytes / int64_t(esize(dtype))
                           : bucket_tile_elems(dtype, N, v8, budgeted(sm_budget));
  const int max_group = std::min(AR_MAX_BUCKET_TENSORS, kMaxBucketPtrs / N);
  static thread_local BucketFusedParams bp;
  std::memset(&bp, 0, sizeof(bp));
  int nt = 0, tiles = 0;
  auto flush = [&]() -> ar_status {
    if (bp.n_seg == 0) {
      nt = 0;
      return AR_OK;
    }
    bp.n = N;
    bp.scale = scale;
    bp.tile_start[bp.n_seg] = tiles;
    const cudaError_t e = tma ? launch_bucket_tma(bp, dtype, stages, tile_bytes, sm_budget, static_cast<cudaStream_t>(stream))
                              : launch_bucket_fused(bp, dtype, sm_budget, v8, static_cast<cudaStream_t>(stream));
    std::memset(&bp, 0, sizeof(bp));
    nt = 0;
    tiles = 0;
    return from_cuda(e);
  };
  for (int t = t_end - 1; t >= t_begin; --t) {  // packing order
    const int64_t o = off[t - t_begin], n_el = int64_t(counts[t]);
    if (n_el == 0) continue;
    // the ring's chunks that overlap this tensor's packed range
    int n_pieces = 0;
    for (int c = 0; c < N; ++c)
      if (std::max(b[c], o) < std::min(b[c + 1], o + n_el)) ++n_pieces;
    if (nt == max_group || bp.n_seg + n_pieces > kMaxBucketSegs) {
      s = flush();
      if (s != AR_OK) return s;
    }
    for (int r = 0; r < N; ++r) bp.ptr[nt * N + r] = tensors[size_t(r) * n_tensors + t];
    for (int c = 0; c < N; ++c) {
      const int64_t lo = std::max(b[c], o), hi = std::min(b[c + 1], o + n_el);
      if (lo >= hi) continue;
      BucketSeg& sg = bp.seg[bp.n_seg];
      sg.t = nt;
      sg.rot = c;
      sg.lo = lo - o;
      sg.hi = hi - o;
      bp.tile_start[bp.n_seg] = tiles;
      const int64_t body = std::max<int64_t>(rdown(sg.hi, W) - rup(sg.lo, W), 0);
      tiles += int(std::max<int64_t>(1, (body + tile - 1) / tile));
      ++bp.n_seg;
    }
    ++nt;
  }
  return flush();
}

// ---------------------------------------------------------------- compression

namespace {

bool valid_block(int block) {
  return block >= AR_COMPRESS_MIN_BLOCK && block <= AR_COMPRESS_MAX_BLOCK && (block & (block - 1)) == 0;
}

size_t n_scale_blocks(size_t count, int block) { return (count + size_t(block) - 1) / size_t(block); }

// Checks shared by the compression calls: ranks, block, the pointer arrays
// (each pointer non-NULL and 16-byte aligned; residuals may be a NULL array).
ar_status check_compress_common(int n_ranks, int block, const void* const* a, const void* const* b) {
  if (n_ranks < 1 || n_ranks > AR_MAX_RANKS || !valid_block(block)) return AR_EINVAL;
  if (a == nullptr || b == nullptr) return AR_EINVAL;
  for (int r = 0; r < n_ranks; ++r)
    if (check_ptr(a[r]) != AR_OK || check_ptr(b[r]) != AR_OK) return AR_EINVAL;
  return AR_OK;
}

void add_ranges(std::vector<std::pair<uintptr_t, uintptr_t>>& iv, const void* const* ptrs, int n, size_t bytes) {
  for (int r = 0; r < n; ++r) iv.push_back({uintptr_t(ptrs[r]), uintptr_t(ptrs[r]) + bytes});
}

CompressParams compress_params(int n_ranks, size_t count, int block, float scale) {
  CompressParams p;
  std::memset(&p, 0, sizeof(p));
  p.n = n_ranks;
  p.block = block;
  p.count = int64_t(count);
  p.n_blocks = int64_t(n_scale_blocks(count, block));
  p.scale = scale;
  return p;
}

}  // namespace

ar_status ar_compress_sizes(size_t count, int block, size_t* n_scales, size_t* message_bytes) {
  if (!valid_block(block)) return AR_EINVAL;
  const size_t nb = n_scale_blocks(count, block);
  if (n_scales != nullptr) *n_scales = nb;
  if (message_bytes != nullptr) *message_bytes = count + 4 * nb;
  return AR_OK;
}

ar_status ar_compress(int n_ranks, size_t count, int block, ar_dtype dtype, const void* const* grads,
                      void* const* residuals, void* const* codes, void* const* scales, void* stream) {
  ar_status s = check_compress_common(n_ranks, block, grads, codes);
  if (s != AR_OK) return s;
  if (dtype != AR_F32 && dtype != AR_BF16) return AR_EINVAL;
  if (scales == nullptr) return AR_EINVAL;
  for (int r = 0; r < n_ranks; ++r) {
    if (check_ptr(scales[r]) != AR_OK) return AR_EINVAL;
    if (residuals != nullptr && check_ptr(residuals[r]) != AR_OK) return AR_EINVAL;
  }
  if (count == 0) return AR_OK;
  std::vector<std::pair<uintptr_t, uintptr_t>> iv;
  add_ranges(iv, grads, n_ranks, count * esize(dtype));
  add_ranges(iv, codes, n_ranks, count);
  add_ranges(iv, scales, n_ranks, 4 * n_scale_blocks(count, block));
  if (residuals != nullptr) add_ranges(iv, residuals, n_ranks, 4 * count);
  if (!disjoint(iv)) return AR_EINVAL;
  CompressParams p = compress_params(n_ranks, count, block, 1.0f);
  p.ef = residuals != nullptr;
  for (int r = 0; r < n_ranks; ++r) {
    p.g[r] = grads[r];
    p.q[r] = static_cast<int8_t*>(codes[r]);
    p.s[r] = static_cast<float*>(scales[r]);
    p.e[r] = residuals != nullptr ? static_cast<float*>(residuals[r]) : nullptr;
  }
  return from_cuda(launch_compress(p, dtype, static_cast<cudaStream_t>(stream)));
}

ar_status ar_compressed_reduce(int n_ranks, size_t count, int block, const void* const* codes,
                               const void* const* scales, float scale, ar_dtype out_dtype, void* const* outs,
                               void* stream) {
  ar_status s = check_compress_common(n_ranks, block, codes, scales);
  if (s != AR_OK) return s;
  if (out_dtype != AR_F32 && out_dtype != AR_BF16) return AR_EINVAL;
  if (!std::isfinite(scale) || outs == nullptr) return AR_EINVAL;
  for (int r = 0; r < n_ranks; ++r)
    if (check_ptr(outs[r]) != AR_OK) return AR_EINVAL;
  if (count == 0) return AR_OK;
  std::vector<std::pair<uintptr_t, uintptr_t>> iv;
  add_ranges(iv, codes, n_ranks, count);
  add_ranges(iv, scales, n_ranks, 4 * n_scale_blocks(count, block));
  add_ranges(iv, outs, n_ranks, count * esize(out_dtype));
  if (!disjoint(iv)) return AR_EINVAL;
  CompressParams p = compress_params(n_ranks, count, block, scale);
  for (int r = 0; r < n_ranks; ++r) {
    p.q[r] = static_cast<int8_t*>(const_cast<void*>(codes[r]));
    p.s[r] = static_cast<float*>(const_cast<void*>(scales[r]));
    p.out[r] = outs[r];
  }
  return from_cuda(launch_compressed_reduce(p, out_dtype, static_cast<cudaStream_t>(stream)));
}

ar_status ar_compressed_allreduce(int n_ranks, size_t count, int block, ar_dtype dtype, const void* const* grads,
                                  void* const* residuals, float scale, void* const* outs, void* stream) {
  if (outs == nullptr) outs = const_cast<void* const*>(grads);  // in place
  ar_status s = check_compress_common(n_ranks, block, grads, outs);
  if (s != AR_OK) return s;
  if (dtype != AR_F32 && dtype != AR_BF16) return AR_EINVAL;
  if (!std::isfinite(scale)) return AR_EINVAL;
  if (residuals != nullptr)
    for (int r = 0; r < n_ranks; ++r)
      if (check_ptr(residuals[r]) != AR_OK) return AR_EINVAL;
  if (count == 0) return AR_OK;
  std::vector<std::pair<uintptr_t, uintptr_t>> iv;
  const size_t bytes = count * esize(dtype);
  add_ranges(iv, grads, n_ranks, bytes);
  for (int r = 0; r < n_ranks; ++r)
    if (outs[r] != grads[r]) iv.push_back({uintptr_t(outs[r]), uintptr_t(outs[r]) + bytes});
  if (residuals != nullptr) add_ranges(iv, residuals, n_ranks, 4 * count);
  if (!disjoint(iv)) return AR_EINVAL;
  CompressParams p = compress_params(n_ranks, count, block, scale);
  p.ef = residuals != nullptr;
  for (int r = 0; r < n_ranks; ++r) {
    p.g[r] = grads[r];
    p.out[r] = outs[r];
    p.e[r] = residuals != nullptr ? static_cast<float*>(residuals[r]) : nullptr;
  }
  return from_cuda(launch_compressed_allreduce(p, dtype, static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------- status

ar_status ar_device_status(int clear) {
  unsigned int v = 0;
  if (read_device_status(&v, clear != 0) != cudaSuccess) return AR_ECUDA;
  return v != 0 ? AR_ETIMEOUT : AR_OK;
}

ar_status ar_plan_query(const ar_plan_t* plan) {
  if (plan == nullptr) return AR_EINVAL;
  const volatile unsigned int* word = host_status_word_if_ready(plan->last_device.v.load(std::memory_order_relaxed));
  return word != nullptr && *word != 0 ? AR_ETIMEOUT : AR_OK;
}

ar_status ar_selftest_wait_timeout(unsigned int polls, void* stream) {
  if (polls == 0) return AR_EINVAL;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return AR_ECUDA;
  volatile unsigned int* word = nullptr;
  if (host_status_word(dev, &word) != cudaSuccess) return AR_ECUDA;  // so that the timeout reaches the host copy
  return from_cuda(launch_wait_timeout(polls, static_cast<cudaStream_t>(stream)));
}

ar_status ar_selftest_scale_quotient(unsigned long long* mismatches) {
  if (mismatches == nullptr) return AR_EINVAL;
  return from_cuda(selftest_div127(mismatches));
}

const char* ar_status_string(ar_status status) {
  switch (status) {
    case AR_OK: return "AR_OK: success";
    case AR_EINVAL: return "AR_EINVAL: invalid argument";
    case AR_EUNSUPPORTED: return "AR_EUNSUPPORTED: not supported by the library";
    case AR_ENOMEM: return "AR_ENOMEM: host allocation failed";
    case AR_ECUDA: return "AR_ECUDA: CUDA runtime error";
    case AR_ETIMEOUT: return "AR_ETIMEOUT: a device-side wait ran out of time";
  }
  return "unknown ar_status";
}

int ar_version(void) { return kVersion; }

}  // extern "C"
