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
// drew (RheoSampling, Key design 2).  Selections count, for each candidate,
// how many keys beat it; the keys are distinct, so the counts are the ranks.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "st_common.cuh"
#include "st_kernels.h"

namespace st {

constexpr int RANK_THREADS = 512;

struct RankShared {
  uint64_t key[SPEC_TREE_MAX_CAND];
  float score[SPEC_TREE_MAX_CAND];
  int32_t token[SPEC_TREE_MAX_CAND];
  int32_t parent[SPEC_TREE_MAX_CAND];  // candidate index of the parent, -1 = root
  int32_t meta[SPEC_TREE_MAX_CAND];    // depth << 16 | kind << 12 | slot
  int32_t exp_row[SPEC_TREE_MAX_CAND];
  int32_t pos[SPEC_TREE_MAX_CAND];     // canonical node index, -1 = pruned
  int32_t aux[SPEC_TREE_MAX_CAND];     // SMART: layer order
  uint64_t skey[SPEC_TREE_MAX_CAND];   // top-R: keys sorted descending
  int32_t sidx[SPEC_TREE_MAX_CAND];    // top-R: candidate of each sorted key
  int32_t front[SPEC_TREE_MAX_NODES];  // current frontier / active list (candidate indices)
  int32_t front_next[SPEC_TREE_MAX_NODES];
  // children of every expanded row, precomputed: entry row * K + slot
  float ch_lp[SPEC_TREE_MAX_CAND];
  int32_t ch_tok[SPEC_TREE_MAX_CAND];
  int32_t ch_kind[SPEC_TREE_MAX_CAND];
  int nc;
  int nf;
  int n_kept;
  int layer_kept;
  int stop;
};

__device__ __forceinline__ uint64_t rank_key(float score, int depth, int prank, int slot) {
  const uint32_t creation = (static_cast<uint32_t>(depth) << 24) | (static_cast<uint32_t>(prank) << 12) |
                            static_cast<uint32_t>(slot);
  return (static_cast<uint64_t>(__float_as_uint(score)) << 32) | (0xffffffffu - creation);
}

// Child `slot` of the node expanded from support row `row` (RheoSampling,
// Key design 2): DET ranks 0..m-1, the probe at slot m with the proxy
// min{q(x_m), z} (q(x_1) + 1 ulp when m = 0), then fillers in rank order
// skipping the probe.  Writes the support rank and returns the local
// probability used for the path score.
__device__ __forceinline__ float child_of(const spec_tree_t& t, int64_t row, int m, int slot, int& kind,
                                          int& rank) {
  const int pp = t.probe_pos[row];
  const float* q = t.sup_q + row * t.sup_stride;
  if (slot < m) {
    kind = SPEC_TREE_DET;
    rank = slot;
    return q[slot];
  }
  if (slot == m && pp >= 0) {
    kind = SPEC_TREE_PROBE;
    rank = pp;
    return m >= 1 ? fminf(q[m - 1], t.sup_z[row]) : nextafterf(q[0], INFINITY);
  }
  kind = SPEC_TREE_FILL;
  const int j = slot - m - (pp >= 0 ? 1 : 0);
  rank = m + j;
  if (pp >= 0 && rank >= pp) ++rank;
  return q[rank];
}

// Children of the first `rows` expanded rows of tree b into shared memory
// (one parallel pass over global memory; the layer loop then reads smem only).
__device__ void load_children(RankShared& s, const RankLaunch& L, int b, int rows) {
  const int K = L.p.K, m = L.p.m;
  const spec_tree_t& t = L.tree;
  for (int idx = threadIdx.x; idx < rows * K; idx += RANK_THREADS) {
    const int r = idx / K, slot = idx - r * K;
    const int64_t row = static_cast<int64_t>(b) * t.n_rows + r;
    int kind, rank;
    s.ch_lp[idx] = child_of(t, row, m, slot, kind, rank);
    s.ch_kind[idx] = kind;
    s.ch_tok[idx] = t.sup_id[row * t.sup_stride + rank];
  }
}

// Generate the K children of every node in s.front[0..nf) at `depth`,
// appending candidates at `base`.  Parent scores come from s.score (root: 1).
__device__ void gen_layer(RankShared& s, const RankLaunch& L, int depth, int nf, int base) {
  const int K = L.p.K;
  for (int idx = threadIdx.x; idx < nf * K; idx += RANK_THREADS) {
    const int f = idx / K, slot = idx - f * K;
    const int pc = s.front[f];
    const int prow = pc < 0 ? 0 : s.exp_row[pc];
    const float pscore = pc < 0 ? 1.0f : s.score[pc];
    const int ci = prow * K + slot;
    const float sc = pscore * s.ch_lp[ci];
    const int c = base + idx;
    s.score[c] = sc;
    s.key[c] = rank_key(sc, depth, f, slot);
    s.token[c] = s.ch_tok[ci];
    s.parent[c] = pc;
    s.meta[c] = (depth << 16) | (s.ch_kind[ci] << 12) | slot;
    s.exp_row[c] = -1;
    s.pos[c] = -1;
  }
}

__device__ void write_nodes(RankShared& s, const RankLaunch& L, int b, int n_nodes) {
  const spec_tree_t& t = L.tree;
  const int64_t nb = static_cast<int64_t>(b) * t.max_nodes;
  for (int i = threadIdx.x; i < t.max_nodes; i += RANK_THREADS) {
    t.node_token[nb + i] = -1;
    t.node_parent[nb + i] = -1;
    t.node_depth[nb + i] = i == 0 ? 0 : -1;
    t.node_kind[nb + i] = i == 0 ? SPEC_TREE_ROOT : -1;
    t.node_slot[nb + i] = -1;
    t.node_exp_row[nb + i] = i == 0 ? 0 : -1;
    t.node_score[nb + i] = i == 0 ? 1.0f : 0.0f;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < s.nc; c += RANK_THREADS) {
    const int pos = s.pos[c];
    if (pos < 0) continue;
    const int pc = s.parent[c];
    t.node_token[nb + pos] = s.token[c];
    t.node_parent[nb + pos] = pc < 0 ? 0 : s.pos[pc];
    t.node_depth[nb + pos] = s.meta[c] >> 16;
    t.node_kind[nb + pos] = (s.meta[c] >> 12) & 0xf;
    t.node_slot[nb + pos] = s.meta[c] & 0xfff;
    t.node_exp_row[nb + pos] = s.exp_row[c];
    t.node_score[nb + pos] = s.score[c];
  }
  if (threadIdx.x == 0) t.n_nodes[b] = n_nodes;
}

// Expand-then-rerank with a frontier of width W per layer, then global top-R.
__global__ void __launch_bounds__(RANK_THREADS) rank_topr_kernel(RankLaunch L) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RankShared& s = *reinterpret_cast<RankShared*>(smem_raw);
  const int b = blockIdx.x, tid = threadIdx.x;
  const int K = L.p.K, W = L.p.W, D = L.p.depth, R = L.p.R;
  load_children(s, L, b, static_cast<int>(L.rows_avail));
  if (tid == 0) {
    s.front[0] = -1;
    s.nf = 1;
    s.nc = 0;
  }
  __syncthreads();
  for (int d = 1; d <= D; ++d) {
    const int nf = s.nf, base = s.nc, ln = nf * K;
    gen_layer(s, L, d, nf, base);
    __syncthreads();
    if (d < D) {
      // frontier of layer d: its top-W candidates, expanded from rows 1 + (d-1)*W + rank
      for (int i = tid; i < ln; i += RANK_THREADS) {
        const uint64_t k = s.key[base + i];
        int r = 0;
        for (int j = 0; j < ln; ++j) r += s.key[base + j] > k;
        if (r < W) {
          s.front_next[r] = base + i;
          s.exp_row[base + i] = 1 + (d - 1) * W + r;
        }
      }
      __syncthreads();
      const int nf2 = ln < W ? ln : W;
      for (int i = tid; i < nf2; i += RANK_THREADS) s.front[i] = s.front_next[i];
      if (tid == 0) {
        s.nf = nf2;
        s.nc = base + ln;
      }
    } else if (tid == 0) {
      s.nc = base + ln;
    }
    __syncthreads();
  }
  const int nc = s.nc;
  // global top-R: bitonic sort of all candidate keys, descending (keys are
  // distinct; the zero padding sorts below every real key)
  int n2 = 1;
  while (n2 < nc) n2 <<= 1;
  for (int i = tid; i < n2; i += RANK_THREADS) {
    s.skey[i] = i < nc ? s.key[i] : 0ull;
    s.sidx[i] = i < nc ? i : -1;
  }
  __syncthreads();
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < n2; i += RANK_THREADS) {
        const int l = i ^ j;
        if (l > i) {
          const uint64_t x = s.skey[i], y = s.skey[l];
          if (((i & k) == 0) ? (x < y) : (x > y)) {
            s.skey[i] = y;
            s.skey[l] = x;
            const int xi = s.sidx[i];
            s.sidx[i] = s.sidx[l];
            s.sidx[l] = xi;
          }
        }
      }
      __syncthreads();
    }
  }
  // canonical order of the top R: depth ascending, then key (sorted order)
  const int nsel = nc < R ? nc : R;
  for (int r = tid; r < nsel; r += RANK_THREADS) {
    const int ci = s.sidx[r];
    const int di = s.meta[ci] >> 16;
    int pos = 1;
    for (int j = 0; j < nsel; ++j) {
      const int dj = s.meta[s.sidx[j]] >> 16;
      pos += (dj < di) || (dj == di && j < r);
    }
    s.pos[ci] = pos;
  }
  __syncthreads();
  write_nodes(s, L, b, 1 + (nc < R ? nc : R));
}

// SMART: layer-wise greedy keep rule over dual-identity children.
// C(n) = 1 + lambda*n + beta + gamma*(exp(delta*n^rho) - 1) + eta (one target
// step included), dC(n) = lambda + gamma*delta*rho*n^(rho-1)*exp(delta*n^rho),
// keep iff alpha*(P(u)/|P|)/dC(n) > L/C(n), with L = 1 + sum of kept P and
// |P| the number of leaves.
__device__ __forceinline__ double smart_cost(double n, const spec_tree_params& p) {
  return 1.0 + p.lambda * n + p.beta + p.gamma * (exp(p.delta * pow(n, (double)p.rho)) - 1.0) + p.eta;
}

__device__ __forceinline__ double smart_dcost(double n, const spec_tree_params& p) {
  const double powterm = n == 0.0 ? 0.0 : p.rho * pow(n, (double)p.rho - 1.0);
  return p.lambda + p.gamma * p.delta * powterm * exp(p.delta * pow(n, (double)p.rho));
}

__global__ void __launch_bounds__(RANK_THREADS) rank_smart_kernel(RankLaunch L) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RankShared& s = *reinterpret_cast<RankShared*>(smem_raw);
  const int b = blockIdx.x, tid = threadIdx.x;
  const int K = L.p.K, D = L.p.depth, budget = L.p.R;
  // per-candidate scratch reused: exp_row doubles as "has a kept child" flag
  // for kept nodes via the high bit of meta (bit 30).
  load_children(s, L, b, static_cast<int>(L.rows_avail));
  if (tid == 0) {
    s.front[0] = -1;
    s.nf = 1;
    s.nc = 0;
    s.n_kept = 0;
    s.stop = 0;
  }
  __syncthreads();
  // state kept by thread 0
  double Lacc = 1.0;
  int paths = 1;
  bool root_has_child = false;
  int next_row = 1;
  for (int d = 1; d <= D; ++d) {
    const int nf = s.nf, base = s.nc, ln = nf * K;
    if (base + ln > SPEC_TREE_MAX_CAND) {
      if (tid == 0) set_status(L.status, SPEC_TREE_S_ROWS);
      break;
    }
    gen_layer(s, L, d, nf, base);
    __syncthreads();
    // order of the layer by key: aux[r] = candidate of rank r
    for (int i = tid; i < ln; i += RANK_THREADS) {
      const uint64_t k = s.key[base + i];
      int r = 0;
      for (int j = 0; j < ln; ++j) r += s.key[base + j] > k;
      s.aux[r] = base + i;
    }
    __syncthreads();
    if (tid == 0) {
      // visit the candidates in key order
      int kept_layer = 0;
      for (int r = 0; r < ln; ++r) {
        if (s.n_kept >= budget) break;
        const int c = s.aux[r];
        const double n = s.n_kept;
        const double lhs = (double)L.p.alpha * ((double)s.score[c] / paths) / smart_dcost(n, L.p);
        const double rhs = Lacc / smart_cost(n, L.p);
        if (lhs > rhs) {
          const int pc = s.parent[c];
          bool parent_has = pc < 0 ? root_has_child : ((s.meta[pc] >> 30) & 1);
          if (parent_has) ++paths;
          if (pc < 0) root_has_child = true;
          else s.meta[pc] |= 1 << 30;
          s.pos[c] = 1 + s.n_kept;  // canonical index = keep order
          s.front_next[kept_layer++] = c;
          s.n_kept += 1;
          Lacc += s.score[c];
        }
      }
      s.layer_kept = kept_layer;
      s.nc = base + ln;
      if (kept_layer == 0 || s.n_kept >= budget || d == D) {
        s.stop = 1;
      } else {
        for (int i = 0; i < kept_layer; ++i) {
          const int c = s.front_next[i];
          if (next_row >= L.rows_avail) {
            set_status(L.status, SPEC_TREE_S_ROWS);
            s.stop = 1;
            break;
          }
          s.exp_row[c] = next_row++;
          s.front[i] = c;
        }
        s.nf = kept_layer;
      }
    }
    __syncthreads();
    if (s.stop) break;
  }
  // clear the helper bit before writing kinds
  for (int c = tid; c < s.nc; c += RANK_THREADS) s.meta[c] &= ~(1 << 30);
  __syncthreads();
  write_nodes(s, L, b, 1 + s.n_kept);
}

cudaError_t launch_rank_topr(const RankLaunch& L, cudaStream_t stream) {
  if (L.B == 0) return cudaSuccess;
  const int smem = static_cast<int>(sizeof(RankShared));
  cudaError_t err = cudaFuncSetAttribute(rank_topr_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  rank_topr_kernel<<<L.B, RANK_THREADS, smem, stream>>>(L);
  return cudaGetLastError();
}

cudaError_t launch_rank_smart(const RankLaunch& L, cudaStream_t stream) {
  if (L.B == 0) return cudaSuccess;
  const int smem = static_cast<int>(sizeof(RankShared));
  cudaError_t err = cudaFuncSetAttribute(rank_smart_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  rank_smart_kernel<<<L.B, RANK_THREADS, smem, stream>>>(L);
  return cudaGetLastError();
}

}  // namespace st
