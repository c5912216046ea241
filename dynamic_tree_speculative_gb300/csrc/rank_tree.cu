// Tree building from expanded rows (sm_103a): one CTA per tree.
//
// Top-R builder: RheoSampling notes, Method / overall framework (cumulative
// path scores, expand-then-rerank, global top-R pruning).  SMART builder:
// SMART notes, Method / Key designs 1-3 and the flowchart (layer-wise greedy
// keep rule alpha * dL/dC > L / C).
//
// Candidates are ranked on a 64-bit key: the float32 score bits in the high
// word (scores are >= 0, so the bit pattern orders them) and the complement
// of the creation index (depth, parent rank, slot) in the low word.  No token
// id enters the key, so a probe's survival never depends on which token it
// drew (RheoSampling, Key design 2).  Keys are distinct, so a key's rank is
// the number of keys above it.
//
// The work per tree is small and sequential in depth, so the kernel is built
// for latency.  Measured on GB300: a dependent shared load costs about 20
// cycles, and several lanes of a warp reading different 16-byte words of one
// bank group cost about 40 more; a shuffle about 30; a ballot with its
// popcount about 70; a global load about a microsecond.  Hence:
//   - every local probability the layers can use is gathered from global
//     memory up front in one round of independent loads (a filler's support
//     rank is slot - 1 or slot, so nothing waits on the probe position); the
//     token ids, which only the written nodes need, are loaded in the same
//     round and land while the layers run;
//   - a layer costs one CTA barrier.  Every candidate of the layer is ranked
//     inside the layer by a group of g lanes: lane p of the group compares
//     against the key pairs p, p + g, p + 2g, ... so that the g lanes read g
//     neighbouring 16-byte words (no bank conflict) in batches of four loads,
//     and the group sums by shuffles.  The rank places the key in the layer's
//     sorted list, and the group of a frontier winner scores that node's
//     children, the next layer's candidates, in the same step;
//   - the global top-R is the head of the merge of the sorted layer lists:
//     a tree of pairwise merges, each cut to R entries, where every output
//     position is one thread's merge-path search.  The survivors of a layer
//     are a prefix of its sorted list, so a survivor's canonical position
//     (depth, then key) is the number of survivors in shallower layers plus
//     its rank in its own layer.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "st_common.cuh"
#include "st_kernels.h"

namespace st {

constexpr int RANK_THREADS = 512;
constexpr int RK_PER_THREAD = (SPEC_TREE_MAX_CAND + RANK_THREADS - 1) / RANK_THREADS;
constexpr int RK_MAX_LAYERS = 256;  // depth <= 255

struct RankShared {
  alignas(16) uint64_t key[SPEC_TREE_MAX_CAND];  // ranking key of every candidate, by creation
  uint64_t mkey[2][SPEC_TREE_MAX_CAND];           // sorted lists being merged (keys, descending)
  int32_t mcand[2][SPEC_TREE_MAX_CAND];           // their candidates
  int32_t link[SPEC_TREE_MAX_CAND];    // (parent candidate + 1) | child-table entry << 12
  int16_t lrank[SPEC_TREE_MAX_CAND];   // rank inside the layer
  int16_t exp_row[SPEC_TREE_MAX_CAND]; // draft row the candidate was expanded from, -1 if none
  int16_t pos[SPEC_TREE_MAX_CAND];     // canonical node index, -1 = pruned
  // child table of every expanded row (entry row * K + slot)
  float ch_lp[SPEC_TREE_MAX_CAND];    // local probability used for the path score
  int32_t ch_rk[SPEC_TREE_MAX_CAND];  // support rank (low 16 bits) | kind << 16
  union {
    int32_t ord[SPEC_TREE_MAX_CAND];     // SMART, during the layers: the current layer by rank
    int32_t ch_tok[SPEC_TREE_MAX_CAND];  // after the layers: token id of each child-table entry
  };
  int32_t nodes[SPEC_TREE_MAX_NODES];     // candidate of canonical node i + 1
  int32_t kept[SPEC_TREE_MAX_NODES];      // SMART: kept candidates in keep order
  int32_t front[2][SPEC_TREE_MAX_NODES];  // SMART, layer mode: frontier of the previous / current layer
  float fscore[SPEC_TREE_MAX_NODES];      // layer mode: path scores of the previous frontier
  float cost[SPEC_TREE_MAX_NODES + 1];    // SMART: C(n)
  float dcost[SPEC_TREE_MAX_NODES + 1];   // SMART: C'(n)
  uint8_t has_kid[SPEC_TREE_MAX_CAND];    // SMART: kept node already has a kept child
  int32_t layer_base[RK_MAX_LAYERS + 1];  // first candidate of layer d (d = 1..D), then the total
  int32_t layer_sel[RK_MAX_LAYERS + 1];   // survivors of the global cut in layer d
  int32_t lst_start[2][RK_MAX_LAYERS];    // merge rounds: start of list i
  int32_t lst_len[2][RK_MAX_LAYERS];      //   and its length
  int nf;      // SMART: frontier size
  int n_kept;  // SMART
  int stop;    // SMART
};

// ---------------------------------------------------------------------- keys ---

__device__ __forceinline__ uint64_t rank_key(float score, int depth, int prank, int slot) {
  const uint32_t creation = (static_cast<uint32_t>(depth) << 24) | (static_cast<uint32_t>(prank) << 12) |
                            static_cast<uint32_t>(slot);
  return (static_cast<uint64_t>(__float_as_uint(score)) << 32) | (0xffffffffu - creation);
}

__device__ __forceinline__ uint32_t key_creation(uint64_t key) {
  return 0xffffffffu - static_cast<uint32_t>(key);
}

__device__ __forceinline__ float key_score(uint64_t key) { return __uint_as_float(static_cast<uint32_t>(key >> 32)); }

__device__ __forceinline__ int key_depth(uint64_t key) { return static_cast<int>(key_creation(key) >> 24); }

// Candidate c: child `slot` of parent candidate pc (-1 = root) at `depth`,
// the parent being frontier rank `prank` and expanded from draft row `prow`.
__device__ __forceinline__ void make_candidate(RankShared& s, int c, int pc, float pscore, int prow, int depth,
                                               int prank, int slot, int K) {
  const int ci = prow * K + slot;
  s.key[c] = rank_key(pscore * s.ch_lp[ci], depth, prank, slot);
  s.link[c] = (pc + 1) | (ci << 12);
  s.exp_row[c] = -1;
  s.pos[c] = -1;
}

// ---------------------------------------------------------------- child table ---
// For every expanded row r < rows and slot < K: the local probability,
// support rank, kind and token of child `slot` (RheoSampling, Key design 2):
// DET ranks 0..m-1, the probe at slot m with the proxy min{q(x_m), z}
// (q(x_1) + 1 ulp when m = 0), fillers in rank order skipping the probe.
// All loads are issued before any is used; the token loads stay in flight in
// `tok` and are stored by store_tokens() once the layers are done.
struct PendingTokens {
  int32_t v[RK_PER_THREAD];
};

__device__ __forceinline__ void load_children(RankShared& s, const RankLaunch& L, int b, int row0, int rows,
                                              PendingTokens& tok) {
  const int K = L.p.K, m = L.p.m;
  const spec_tree_t& t = L.tree;
  const int n = rows * K;
  const int e0 = row0 * K;  // child-table entry of the range's first child
  int pp[RK_PER_THREAD];
  float qa[RK_PER_THREAD], qb[RK_PER_THREAD], z[RK_PER_THREAD];
#pragma unroll
  for (int u = 0; u < RK_PER_THREAD; ++u) {
    const int idx = threadIdx.x + u * RANK_THREADS;
    if (idx < n) {
      const int r = row0 + idx / K, slot = idx % K;
      const int64_t row = static_cast<int64_t>(b) * t.n_rows + r;
      const float* q = t.sup_q + row * t.sup_stride;
      pp[u] = t.probe_pos[row];
      qa[u] = q[slot];
      qb[u] = slot > 0 ? q[slot - 1] : 0.0f;
      z[u] = t.sup_z[row];
    }
  }
#pragma unroll
  for (int u = 0; u < RK_PER_THREAD; ++u) {
    const int idx = threadIdx.x + u * RANK_THREADS;
    if (idx < n) {
      const int r = row0 + idx / K, slot = idx % K;
      int kind, rank;
      float lp;
      if (slot < m) {
        kind = SPEC_TREE_DET;
        rank = slot;
        lp = qa[u];
      } else if (slot == m && pp[u] >= 0) {
        kind = SPEC_TREE_PROBE;
        rank = pp[u];
        lp = m >= 1 ? fminf(qb[u], z[u]) : nextafterf(qa[u], INFINITY);
      } else {
        // fillers take tail ranks m, m+1, ... skipping the probe's rank
        kind = SPEC_TREE_FILL;
        rank = (pp[u] >= 0 && slot - 1 < pp[u]) ? slot - 1 : slot;
        lp = rank == slot ? qa[u] : qb[u];
      }
      s.ch_lp[e0 + idx] = lp;
      s.ch_rk[e0 + idx] = (rank & 0xffff) | (kind << 16);
      const int64_t row = static_cast<int64_t>(b) * t.n_rows + r;
      // a dense support keeps ranks 0..K-1 and the probe at entry K
      const int entry = kind == SPEC_TREE_PROBE && rank > L.probe_entry_cap ? L.probe_entry_cap : rank;
      tok.v[u] = t.sup_id[row * t.sup_stride + entry];
    }
  }
}

__device__ __forceinline__ void store_tokens(RankShared& s, int row0, int rows, int K, const PendingTokens& tok) {
#pragma unroll
  for (int u = 0; u < RK_PER_THREAD; ++u) {
    const int idx = threadIdx.x + u * RANK_THREADS;
    if (idx < rows * K) s.ch_tok[row0 * K + idx] = tok.v[u];
  }
}

// ------------------------------------------------------------ layer ranking ---

// Four 16-byte shared loads issued back to back.
__device__ __forceinline__ void lds_pairs4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint64_t (&v)[8]) {
  asm volatile(
      "ld.shared.v2.u64 {%0, %1}, [%8];\n\t"
      "ld.shared.v2.u64 {%2, %3}, [%9];\n\t"
      "ld.shared.v2.u64 {%4, %5}, [%10];\n\t"
      "ld.shared.v2.u64 {%6, %7}, [%11];"
      : "=l"(v[0]), "=l"(v[1]), "=l"(v[2]), "=l"(v[3]), "=l"(v[4]), "=l"(v[5]), "=l"(v[6]), "=l"(v[7])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3)
      : "memory");
}

// Number of keys above x among the n keys at s.key[base..), counted by lane
// `part` of a group of g lanes: the keys are read as 16-byte pairs from the
// aligned word below the list, pairs part, part + g, ...; keys outside the
// list are masked.
__device__ __forceinline__ int count_part(const RankShared& s, int base, int n, uint64_t x, int g, int part) {
  const uint32_t k0 = smem_u32(s.key);       // 16-byte aligned
  const int first = base & ~1;               // first key of the first pair
  const int npairs = (base + n - first + 1) >> 1;
  int r = 0;
  int q = part;
  for (; q + 3 * g < npairs; q += 4 * g) {
    uint64_t v[8];
    lds_pairs4(k0 + 8u * (first + 2 * q), k0 + 8u * (first + 2 * (q + g)), k0 + 8u * (first + 2 * (q + 2 * g)),
               k0 + 8u * (first + 2 * (q + 3 * g)), v);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = first + 2 * (q + u * g);
      r += (j >= base && v[2 * u] > x) + (j + 1 < base + n && v[2 * u + 1] > x);
    }
  }
  for (; q < npairs; q += g) {
    const int j = first + 2 * q;
    const uint64_t a = s.key[j];
    const uint64_t b = j + 1 < base + n ? s.key[j + 1] : 0ull;
    r += (j >= base && a > x) + (b > x);
  }
  return r;
}

// Ranks inside the layer of the n keys at s.key[base..base+n): every lane of
// the group ranking key i calls f(i, rank, g, part) with the group size g and
// its lane's place part in the group, so the group can share follow-up work.
// Groups are powers of two up to 32 lanes, as large as the CTA allows; layers
// above RANK_THREADS keys are ranked one thread per key.  All threads call
// it; no barrier inside.
template <typename F>
__device__ __forceinline__ void rank_layer(const RankShared& s, int base, int n, F f) {
  const int tid = threadIdx.x;
  if (n <= RANK_THREADS) {
    int g = 1;
    while (g < 32 && 2 * g * n <= RANK_THREADS) g *= 2;
    const int i = tid / g, part = tid & (g - 1);
    const bool valid = i < n;
    const uint64_t x = valid ? s.key[base + i] : 0xffffffffffffffffull;
    int r = count_part(s, base, n, x, g, part);
    for (int o = 1; o < g; o <<= 1) r += __shfl_xor_sync(FULL, r, o);
    if (valid) f(i, r, g, part);
  } else {
    for (int i = tid; i < n; i += RANK_THREADS) f(i, count_part(s, base, n, s.key[base + i], 1, 0), 1, 0);
  }
}

// ------------------------------------------------------------- merge of lists ---

// Entry p (descending) of the merge of the descending lists a[0..na) and
// b[0..nb) (distinct keys), by a merge-path search: i = how many of the top
// p + 1 entries come from a.
__device__ __forceinline__ void merge_entry(const uint64_t* ka, const int32_t* ca, int na, const uint64_t* kb,
                                            const int32_t* cb, int nb, int p, uint64_t& key, int32_t& cand) {
  int lo = max(0, p - nb), hi = min(p, na);
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (ka[mid] > kb[p - 1 - mid]) lo = mid + 1;
    else hi = mid;
  }
  const int j = p - lo;
  if (j >= nb || (lo < na && ka[lo] > kb[j])) {
    key = ka[lo];
    cand = ca[lo];
  } else {
    key = kb[j];
    cand = cb[j];
  }
}

// Node arrays of tree b: node 0 is the root, node i >= 1 the candidate
// s.nodes[i - 1] (canonical order), unused entries -1 (score 0).
__device__ void write_nodes(RankShared& s, const RankLaunch& L, int b, int nsel) {
  const spec_tree_t& t = L.tree;
  const int64_t nb = static_cast<int64_t>(b) * t.max_nodes;
  for (int i = threadIdx.x; i < t.max_nodes; i += RANK_THREADS) {
    int tok = -1, par = -1, dep = -1, kind = -1, slot = -1, er = -1;
    float sc = 0.0f;
    if (i == 0) {
      dep = 0;
      kind = SPEC_TREE_ROOT;
      er = 0;
      sc = 1.0f;
    } else if (i <= nsel) {
      const int c = s.nodes[i - 1];
      const uint64_t key = s.key[c];
      const uint32_t cr = key_creation(key);
      const int link = s.link[c];
      const int ci = link >> 12, pc = (link & 0xfff) - 1;
      tok = s.ch_tok[ci];
      par = pc < 0 ? 0 : s.pos[pc];
      dep = static_cast<int>(cr >> 24);
      kind = s.ch_rk[ci] >> 16;
      slot = static_cast<int>(cr & 0xfffu);
      er = s.exp_row[c];
      sc = key_score(key);
    }
    t.node_token[nb + i] = tok;
    t.node_parent[nb + i] = par;
    t.node_depth[nb + i] = dep;
    t.node_kind[nb + i] = kind;
    t.node_slot[nb + i] = slot;
    t.node_exp_row[nb + i] = er;
    t.node_score[nb + i] = sc;
  }
  if (threadIdx.x == 0) t.n_nodes[b] = 1 + nsel;
}

// Global top-R of a tree whose D layers are ranked: s.mkey[0] / s.mcand[0]
// hold each layer's sorted list at the layer's base (s.layer_base), s.lrank
// each candidate's rank in its layer, s.lst_start[0] / s.lst_len[0] the
// lists cut to R, s.layer_sel zero.  Sets s.pos and s.nodes of the min(R, nc)
// survivors in canonical order.  Rounds of pairwise merges of the sorted
// layer lists, each cut to R: list i keeps the start of the block of layers
// it covers, and a merge of two neighbours fits in their joint block.  Each
// output entry is one thread's merge-path search.
__device__ void topr_cut(RankShared& s, int D, int R) {
  const int tid = threadIdx.x;
  int nl = D, cur = 0;
  while (nl > 1) {
    const int nl2 = (nl + 1) >> 1;
    const int32_t* st = s.lst_start[cur];
    const int32_t* len = s.lst_len[cur];
    for (int e = tid; e < nl2 * R; e += RANK_THREADS) {
      const int i = e / R, p = e - i * R;
      const int a0 = st[2 * i], la = len[2 * i];
      const bool pair = 2 * i + 1 < nl;
      const int b0 = pair ? st[2 * i + 1] : a0, lb = pair ? len[2 * i + 1] : 0;
      if (p == 0) {
        s.lst_start[cur ^ 1][i] = a0;
        s.lst_len[cur ^ 1][i] = min(R, la + lb);
      }
      if (p < la + lb) {
        uint64_t k;
        int32_t c;
        merge_entry(s.mkey[cur] + a0, s.mcand[cur] + a0, la, s.mkey[cur] + b0, s.mcand[cur] + b0, lb, p, k, c);
        s.mkey[cur ^ 1][a0 + p] = k;
        s.mcand[cur ^ 1][a0 + p] = c;
      }
    }
    __syncthreads();
    nl = nl2;
    cur ^= 1;
  }
  // s.mkey[cur][0..nsel): the top-R by key; survivors per layer
  const int nsel = min(R, s.layer_base[D + 1]);
  for (int p = tid; p < nsel; p += RANK_THREADS) {
    const int c = s.mcand[cur][p];
    s.pos[c] = 0;  // survivor; canonical index set below
    atomicAdd(&s.layer_sel[key_depth(s.key[c])], 1);
  }
  __syncthreads();
  // canonical index: survivors of shallower layers, then rank in the layer
  for (int p = tid; p < nsel; p += RANK_THREADS) {
    const int c = s.mcand[cur][p];
    const int d = key_depth(s.key[c]);
    int q = 1 + s.lrank[c];
    for (int e = 1; e < d; ++e) q += s.layer_sel[e];
    s.pos[c] = static_cast<int16_t>(q);
    if (q - 1 < SPEC_TREE_MAX_NODES) s.nodes[q - 1] = c;
  }
}


// Expand-then-rerank with a frontier of width W per layer, then global top-R.
__global__ void __launch_bounds__(RANK_THREADS) rank_topr_kernel(RankLaunch L) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RankShared& s = *reinterpret_cast<RankShared*>(smem_raw);
  const int b = blockIdx.x, tid = threadIdx.x;
  const int K = L.p.K, W = L.p.W, D = L.p.depth, R = L.p.R;
  const int rows = static_cast<int>(L.rows_avail);
  grid_dependency_wait();  // the support arrays come from the previous kernel
  PendingTokens tok;
  load_children(s, L, b, 0, rows, tok);
  // layer sizes: K, then min(previous, W) * K; each sorted layer list is
  // list d - 1 of the merge tree
  if (tid == 0) {
    int base = 0, ln = K;
    for (int d = 1; d <= D; ++d) {
      s.layer_base[d] = base;
      s.lst_start[0][d - 1] = base;
      s.lst_len[0][d - 1] = min(R, ln);  // only a layer's first R can survive
      base += ln;
      ln = (ln < W ? ln : W) * K;
    }
    s.layer_base[D + 1] = base;
  }
  if (tid <= D) s.layer_sel[tid] = 0;
  __syncthreads();
  // layer 1: the root's children
  for (int slot = tid; slot < K; slot += RANK_THREADS) make_candidate(s, slot, -1, 1.0f, 0, 1, 0, slot, K);
  __syncthreads();
  for (int d = 1; d <= D; ++d) {
    const int base = s.layer_base[d], ln = s.layer_base[d + 1] - base;
    const int next = s.layer_base[d + 1];
    const int row0 = 1 + (d - 1) * W;
    // rank the layer into its sorted list; frontier rank r < W is expanded
    // from draft row row0 + r and its group scores the K children
    rank_layer(s, base, ln, [&](int i, int r, int g, int part) {
      const int c = base + i;
      const uint64_t key = s.key[c];
      if (part == 0) {
        s.lrank[c] = static_cast<int16_t>(r);
        s.mkey[0][base + r] = key;
        s.mcand[0][base + r] = c;
      }
      if (d < D && r < W) {
        const int prow = row0 + r;
        if (part == 0) s.exp_row[c] = static_cast<int16_t>(prow);
        const float ps = key_score(key);
        for (int slot = part; slot < K; slot += g)
          make_candidate(s, next + r * K + slot, c, ps, prow, d + 1, r, slot, K);
      }
    });
    __syncthreads();
  }
  grid_dependents_launch();
  topr_cut(s, D, R);
  store_tokens(s, 0, rows, K, tok);
  __syncthreads();
  write_nodes(s, L, b, min(R, s.layer_base[D + 1]));
}

// SMART: layer-wise greedy keep rule over dual-identity children.
// C(n) = 1 + lambda*n + beta + gamma*(exp(delta*n^rho) - 1) + eta (one target
// step included), C'(n) = lambda + gamma*delta*rho*n^(rho-1)*exp(delta*n^rho)
// (the n^(rho-1) term is 0 at n = 0), keep iff alpha*(P(u)/|P|)/C'(n) > L/C(n),
// with L = 1 + sum of kept P and |P| the number of leaves.
//
// Within a layer the candidates are visited in descending key and the state
// (n, L, |P|) changes only on a keep, so the left side can only fall and the
// right side only rise along the layer: after the first rejection no later
// candidate of the layer can be kept, and the scan stops there.
__device__ __forceinline__ float smart_cost_f(int n, const spec_tree_params& p) {
  const float nr = n == 0 ? 0.0f : powf(static_cast<float>(n), p.rho);
  return 1.0f + p.lambda * n + p.beta + p.gamma * (expf(p.delta * nr) - 1.0f) + p.eta;
}

__device__ __forceinline__ float smart_dcost_f(int n, const spec_tree_params& p) {
  if (n == 0) return p.lambda;
  const float nf = static_cast<float>(n);
  return p.lambda + p.gamma * p.delta * p.rho * powf(nf, p.rho - 1.0f) * expf(p.delta * powf(nf, p.rho));
}

__global__ void __launch_bounds__(RANK_THREADS) rank_smart_kernel(RankLaunch L) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RankShared& s = *reinterpret_cast<RankShared*>(smem_raw);
  const int b = blockIdx.x, tid = threadIdx.x;
  const int K = L.p.K, D = L.p.depth, budget = L.p.R;
  // cost tables (no dependence on the previous kernel)
  for (int n = tid; n <= budget; n += RANK_THREADS) {
    s.cost[n] = smart_cost_f(n, L.p);
    s.dcost[n] = smart_dcost_f(n, L.p);
  }
  grid_dependency_wait();
  const int rows = static_cast<int>(L.rows_avail);
  PendingTokens tok;
  load_children(s, L, b, 0, rows, tok);
  if (tid == 0) {
    s.front[0][0] = -1;
    s.nf = 1;
    s.n_kept = 0;
    s.stop = 0;
  }
  __syncthreads();
  // state kept by thread 0
  double Lacc = 1.0;
  int paths = 1;
  bool root_has_child = false;
  int next_row = 1;
  int nc = 0, cur = 0;
  for (int d = 1; d <= D; ++d) {
    const int nf = s.nf, base = nc, ln = nf * K;
    if (base + ln > SPEC_TREE_MAX_CAND) {
      if (tid == 0) set_status(L.status, SPEC_TREE_S_ROWS);
      break;
    }
    // candidates: the K children of every node kept in the previous layer
    for (int idx = tid; idx < ln; idx += RANK_THREADS) {
      const int f = idx / K, slot = idx - f * K;
      const int pc = s.front[cur][f];
      const float ps = pc < 0 ? 1.0f : key_score(s.key[pc]);
      const int prow = pc < 0 ? 0 : s.exp_row[pc];
      make_candidate(s, base + idx, pc, ps, prow, d, f, slot, K);
    }
    __syncthreads();
    nc = base + ln;
    // the layer in key order, as far as it can be kept
    const int room = budget - s.n_kept;
    const int need = ln < room + 1 ? ln : room + 1;
    rank_layer(s, base, ln, [&](int i, int r, int, int part) {
      if (part == 0 && r < need) s.ord[base + r] = base + i;
    });
    __syncthreads();
    if (tid == 0) {
      int32_t* fn = s.front[cur ^ 1];
      int kept_layer = 0;
      for (int r = 0; r < need && s.n_kept < budget; ++r) {
        const int c = s.ord[base + r];
        const int n = s.n_kept;
        const float sc = key_score(s.key[c]);
        const float lhs = L.p.alpha * (sc / static_cast<float>(paths)) / s.dcost[n];
        const float rhs = static_cast<float>(Lacc) / s.cost[n];
        if (!(lhs > rhs)) break;
        const int pc = (s.link[c] & 0xfff) - 1;
        const bool parent_has = pc < 0 ? root_has_child : s.has_kid[pc] != 0;
        if (parent_has) ++paths;
        if (pc < 0) root_has_child = true;
        else s.has_kid[pc] = 1;
        s.has_kid[c] = 0;
        s.pos[c] = static_cast<int16_t>(1 + n);  // keep order is the canonical order
        s.kept[n] = c;
        fn[kept_layer++] = c;
        s.n_kept = n + 1;
        Lacc += static_cast<double>(sc);
      }
      if (kept_layer == 0 || s.n_kept >= budget || d == D) {
        s.stop = 1;
      } else {
        for (int i = 0; i < kept_layer; ++i) {
          if (next_row >= rows) {
            set_status(L.status, SPEC_TREE_S_ROWS);
            s.stop = 1;
            break;
          }
          s.exp_row[fn[i]] = static_cast<int16_t>(next_row++);
        }
        s.nf = kept_layer;
      }
    }
    __syncthreads();
    cur ^= 1;
    if (s.stop) break;
  }
  grid_dependents_launch();
  const int nsel = s.n_kept;
  for (int i = tid; i < nsel; i += RANK_THREADS) s.nodes[i] = s.kept[i];
  store_tokens(s, 0, rows, K, tok);
  __syncthreads();
  write_nodes(s, L, b, nsel);
}

// ------------------------------------------------- layer-by-layer builder ---
// The same tree as rank_topr_kernel, built one layer per call so that a draft
// model can produce each frontier's logits in between (RheoSampling notes,
// overall framework: the frontier is expanded layer by layer).  Call `layer`
// (0 .. depth-1) finds the draft rows of the current frontier (layer 0: the
// root) expanded into the tree's support rows; it scores their children, the
// candidates of depth layer + 1, ranks them inside their layer, names the
// next frontier and keeps all of it in a per-tree state in global memory.
// The finish call cuts the global top-R from the state exactly as the
// one-shot build does, so both give the same tree bit for bit.  The state
// holds every candidate's token and kind, so the finish call never reads a
// support row (rows of frontier ranks that did not exist are never written).
struct alignas(16) LayerState {
  int32_t nc;      // candidates so far
  int32_t nf;      // size of the frontier to expand next
  int32_t layers;  // layers ranked so far; -1 after a call out of order
  int32_t pad;
  int32_t front[SPEC_TREE_MAX_NODES];     // candidate of frontier rank r
  int32_t layer_base[RK_MAX_LAYERS + 4];  // first candidate of layer d, then the end
  uint64_t key[SPEC_TREE_MAX_CAND];
  int32_t link[SPEC_TREE_MAX_CAND];
  int32_t ch_rk[SPEC_TREE_MAX_CAND];   // child-table entry: support rank | kind << 16
  int32_t ch_tok[SPEC_TREE_MAX_CAND];  // child-table entry: token id
  int16_t exp_row[SPEC_TREE_MAX_CAND];
  int16_t lrank[SPEC_TREE_MAX_CAND];
};

size_t layer_state_bytes() { return sizeof(LayerState); }

// Frontier outputs of tree b from rank r0 on: none.
__device__ __forceinline__ void clear_frontier(const RankLaunch& L, int b, int r0) {
  const int W = L.p.W;
  for (int r = r0 + static_cast<int>(threadIdx.x); r < W; r += RANK_THREADS) {
    if (L.frontier_token) L.frontier_token[static_cast<int64_t>(b) * W + r] = -1;
    if (L.frontier_parent) L.frontier_parent[static_cast<int64_t>(b) * W + r] = -1;
  }
}

__global__ void __launch_bounds__(RANK_THREADS) layer_topr_kernel(RankLaunch L) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RankShared& s = *reinterpret_cast<RankShared*>(smem_raw);
  const int b = blockIdx.x, tid = threadIdx.x;
  const int K = L.p.K, W = L.p.W, D = L.p.depth;
  const int layer = L.layer, depth = layer + 1;
  const int nf = static_cast<int>(L.rows_avail);  // frontier rows expanded for this call
  LayerState* g = reinterpret_cast<LayerState*>(L.state) + b;
  grid_dependency_wait();  // the support rows (and the state) come from earlier kernels
  const int ln = nf * K;
  const int nc = layer == 0 ? 0 : g->nc;
  // the state must come from the previous layer's call; every index read
  // from it is range-checked, so a spoiled state is never followed
  bool bad = layer > 0 && (g->layers != layer || g->nf != nf || nc < 0 || nc > SPEC_TREE_MAX_CAND - ln);
  const int row0 = layer == 0 ? 0 : 1 + (layer - 1) * W;
  PendingTokens tok;
  load_children(s, L, b, row0, nf, tok);
  if (!bad) {
    for (int f = tid; f < nf; f += RANK_THREADS) {
      const int pc = layer == 0 ? -1 : g->front[f];
      if (layer > 0 && (pc < 0 || pc >= nc)) {
        bad = true;
        break;
      }
      s.front[0][f] = pc;
      s.fscore[f] = pc < 0 ? 1.0f : key_score(g->key[pc]);
    }
  }
  store_tokens(s, row0, nf, K, tok);
  if (__syncthreads_or(bad)) {  // every thread has read the header
    if (tid == 0) {
      g->layers = -1;
      set_status(L.status, SPEC_TREE_S_LAYERS);
    }
    clear_frontier(L, b, 0);
    return;
  }
  for (int idx = tid; idx < ln; idx += RANK_THREADS) {
    const int f = idx / K, slot = idx - f * K;
    make_candidate(s, nc + idx, s.front[0][f], s.fscore[f], row0 + f, depth, f, slot, K);
  }
  __syncthreads();
  const bool more = depth < D;
  const int nf2 = ln < W ? ln : W;
  // rank the layer; its first W are the next frontier, expanded from the
  // draft rows 1 + layer * W + r
  rank_layer(s, nc, ln, [&](int i, int r, int, int part) {
    if (part != 0) return;
    const int c = nc + i;
    s.lrank[c] = static_cast<int16_t>(r);
    if (more && r < W) {
      s.exp_row[c] = static_cast<int16_t>(1 + layer * W + r);
      s.front[1][r] = c;
      const int64_t o = static_cast<int64_t>(b) * W + r;
      if (L.frontier_token) L.frontier_token[o] = s.ch_tok[s.link[c] >> 12];
      if (L.frontier_parent)
        L.frontier_parent[o] = layer == 0 ? -1 : static_cast<int>((key_creation(s.key[c]) >> 12) & 0xfffu);
    }
  });
  __syncthreads();
  grid_dependents_launch();
  for (int idx = tid; idx < ln; idx += RANK_THREADS) {
    const int c = nc + idx, e = row0 * K + idx;
    g->key[c] = s.key[c];
    g->link[c] = s.link[c];
    g->exp_row[c] = s.exp_row[c];
    g->lrank[c] = s.lrank[c];
    g->ch_rk[e] = s.ch_rk[e];
    g->ch_tok[e] = s.ch_tok[e];
  }
  if (more)
    for (int r = tid; r < nf2; r += RANK_THREADS) g->front[r] = s.front[1][r];
  clear_frontier(L, b, more ? nf2 : 0);
  if (tid == 0) {
    g->nc = nc + ln;
    g->nf = more ? nf2 : 0;
    g->layers = depth;
    if (layer == 0) g->layer_base[1] = 0;
    g->layer_base[depth + 1] = nc + ln;
  }
}

__global__ void __launch_bounds__(RANK_THREADS) layer_finish_kernel(RankLaunch L) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RankShared& s = *reinterpret_cast<RankShared*>(smem_raw);
  const int b = blockIdx.x, tid = threadIdx.x;
  const int D = L.p.depth, R = L.p.R;
  const LayerState* g = reinterpret_cast<const LayerState*>(L.state) + b;
  grid_dependency_wait();
  const int nc = g->nc;
  // the state must hold all D layers; every index read from it is
  // range-checked, so a spoiled state is never followed
  bool bad = g->layers != D || nc < 0 || nc > SPEC_TREE_MAX_CAND;
  if (!bad) {
    for (int d = 1 + tid; d <= D + 1; d += RANK_THREADS) s.layer_base[d] = g->layer_base[d];
    for (int c = tid; c < nc; c += RANK_THREADS) {
      s.key[c] = g->key[c];
      s.link[c] = g->link[c];
      s.lrank[c] = g->lrank[c];
      s.exp_row[c] = g->exp_row[c];
      s.pos[c] = -1;
      s.mkey[0][c] = 0;
      s.mcand[0][c] = 0;
    }
    for (int i = tid; i < R; i += RANK_THREADS) s.nodes[i] = 0;
  }
  if (tid <= D) s.layer_sel[tid] = 0;
  if (__syncthreads_or(bad)) {
    // not every layer was ranked, in order: the root alone and a status bit
    if (tid == 0) set_status(L.status, SPEC_TREE_S_LAYERS);
    write_nodes(s, L, b, 0);
    return;
  }
  for (int d = 1 + tid; d <= D; d += RANK_THREADS) {
    const int lo = s.layer_base[d], hi = s.layer_base[d + 1];
    if ((d == 1 && lo != 0) || hi < lo || hi > nc || (d == D && hi != nc)) bad = true;
  }
  for (int c = tid; c < nc; c += RANK_THREADS) {
    const int link = s.link[c], e = link >> 12, pc = (link & 0xfff) - 1, d = key_depth(s.key[c]);
    if (e < 0 || e >= SPEC_TREE_MAX_CAND || pc >= c || d < 1 || d > D || s.lrank[c] < 0 ||
        s.lrank[c] >= s.layer_base[d + 1] - s.layer_base[d]) {
      bad = true;
      continue;
    }
    s.ch_rk[e] = g->ch_rk[e];
    s.ch_tok[e] = g->ch_tok[e];
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) set_status(L.status, SPEC_TREE_S_LAYERS);
    write_nodes(s, L, b, 0);
    return;
  }
  grid_dependents_launch();
  // each layer's sorted list, cut to R, from the ranks kept in the state
  for (int d = 1 + tid; d <= D; d += RANK_THREADS) {
    s.lst_start[0][d - 1] = s.layer_base[d];
    s.lst_len[0][d - 1] = min(R, s.layer_base[d + 1] - s.layer_base[d]);
  }
  for (int c = tid; c < nc; c += RANK_THREADS) {
    const int p = s.layer_base[key_depth(s.key[c])] + s.lrank[c];
    s.mkey[0][p] = s.key[c];
    s.mcand[0][p] = c;
  }
  __syncthreads();
  topr_cut(s, D, R);
  __syncthreads();
  write_nodes(s, L, b, min(R, nc));
}

template <typename Kern>
cudaError_t launch_rank(Kern kern, const RankLaunch& L, cudaStream_t stream) {
  if (L.B == 0) return cudaSuccess;
  const int smem = static_cast<int>(sizeof(RankShared));
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(kern, dim3(L.B), dim3(RANK_THREADS), smem, stream, L);
}

cudaError_t launch_rank_topr(const RankLaunch& L, cudaStream_t stream) {
  return launch_rank(rank_topr_kernel, L, stream);
}

cudaError_t launch_rank_smart(const RankLaunch& L, cudaStream_t stream) {
  return launch_rank(rank_smart_kernel, L, stream);
}

cudaError_t launch_layer_topr(const RankLaunch& L, cudaStream_t stream) {
  return launch_rank(layer_topr_kernel, L, stream);
}

cudaError_t launch_layer_finish(const RankLaunch& L, cudaStream_t stream) {
  return launch_rank(layer_finish_kernel, L, stream);
}

}  // namespace st
