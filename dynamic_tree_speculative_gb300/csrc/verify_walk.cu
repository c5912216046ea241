// Layer-by-layer verification of built trees (sm_103a): one CTA per tree.
//
// RheoSampling notes, Method / Key design 3: the probe is tested first with
// min(1, p/q~_T); on rejection the residual w = max(0, p - q~_T) (w = p off
// the tail) with mass Zr = 1 - sum_tail min(p, q~_T) is used for recursive
// rejection of the remaining children, each a one-hot draft (accept with
// w(x)/Zr, else drop x); the bonus token is drawn from the final residual.
// p = softmax(t / T) over the whole vocabulary of the current node's target
// row (training-strategy paragraph: verification runs at temperature T).
//
// Per level the CTA streams the node's target row once with 16-byte loads for
// the online max / sum-exp, gathers p at the <= |S| support tokens of the
// node's draft row (the tail and the children), and thread 0 takes the
// decisions.  Only the final level streams its row a second time, in token-id
// order, for the bonus inverse CDF (w differs from p only at support tokens,
// which are patched from a small id-sorted list).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "st_common.cuh"
#include "st_kernels.h"

namespace st {

constexpr int VER_THREADS = 1024;
constexpr int VER_WARPS = VER_THREADS / 32;
constexpr float LOG2E = 1.4426950408889634f;
constexpr double MASS_MARGIN = 1e-6;

struct VerShared {
  int32_t node_parent[SPEC_TREE_MAX_NODES];
  int32_t kids[SPEC_TREE_MAX_SUPPORT];  // children of the current node (node indices)
  int nkids;
  float p_sup[SPEC_TREE_MAX_SUPPORT];   // p at support ranks of the node's draft row
  float qt_sup[SPEC_TREE_MAX_SUPPORT];  // q~_T at support ranks (0 off the tail)
  float w_sup[SPEC_TREE_MAX_SUPPORT];   // residual at support ranks
  int32_t corr_id[SPEC_TREE_MAX_SUPPORT];  // id-sorted tokens whose w differs from p
  float corr_w[SPEC_TREE_MAX_SUPPORT];
  int ncorr;
  float red_m[VER_WARPS];
  float red_s[VER_WARPS];
  float scan_w[VER_WARPS];
  float scan_x[VER_WARPS];
  float chunk_total;
  float target_rel;
  double running;
  float M;       // max logit of the row
  double Zp;     // sum of exp2((t - M) * log2e / T)
  double Zr;     // residual mass
  int accepted;  // accepted child node or -1
  int residual;  // probe rejected: tail residual in force
  int bonus;
  int bonus_last;
};

template <typename T>
struct VElem;
template <>
struct VElem<__nv_bfloat16> {
  static constexpr int VEC = 8, ES = 2;
  __device__ static float get(const uint4& v, int j) {
    const uint32_t w = (j < 2) ? v.x : (j < 4) ? v.y : (j < 6) ? v.z : v.w;
    return __uint_as_float(((w >> (16 * (j & 1))) & 0xffffu) << 16);
  }
  __device__ static float load(const uint8_t* row, int v) {
    return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(row)[v]) << 16);
  }
};
template <>
struct VElem<float> {
  static constexpr int VEC = 4, ES = 4;
  __device__ static float get(const uint4& v, int j) {
    return __uint_as_float((j == 0) ? v.x : (j == 1) ? v.y : (j == 2) ? v.z : v.w);
  }
  __device__ static float load(const uint8_t* row, int v) { return reinterpret_cast<const float*>(row)[v]; }
};

// Block-wide max and sum-exp of one row: M = max t, Zp = sum exp2((t - M) * c),
// c = log2(e) / T.  Online per thread (rescale when the running max grows),
// compensated float32 accumulation per thread, float64 across threads.
template <typename T>
__device__ void row_stats(VerShared& s, const uint8_t* row, int V, float c, bool& nonfinite) {
  using E = VElem<T>;
  constexpr int VEC = E::VEC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nvec = static_cast<int>((static_cast<int64_t>(V) * E::ES) / 16);
  float m_run = -INFINITY, s_run = 0.0f, comp = 0.0f;
  auto consume = [&](const float* x, int n) {
    float vmax = -INFINITY;
    for (int j = 0; j < n; ++j) vmax = fmaxf(vmax, x[j]);
    for (int j = 0; j < n; ++j)
      if (!(x[j] == x[j]) || x[j] == INFINITY) nonfinite = true;
    if (vmax == -INFINITY || !(vmax == vmax)) return;
    if (vmax > m_run) {
      const float f = exp2f((m_run - vmax) * c);
      s_run *= f;
      comp *= f;
      m_run = vmax;
    }
    float vs = 0.0f;
    for (int j = 0; j < n; ++j) vs += exp2f((x[j] - m_run) * c);
    const float y = vs - comp;
    const float t = s_run + y;
    comp = (t - s_run) - y;
    s_run = t;
  };
  const uint4* rv = reinterpret_cast<const uint4*>(row);
  int i = tid;
  for (; i + 3 * VER_THREADS < nvec; i += 4 * VER_THREADS) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = ldg_stream(rv + i + u * VER_THREADS);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float x[VEC];
#pragma unroll
      for (int j = 0; j < VEC; ++j) x[j] = E::get(v[u], j);
      consume(x, VEC);
    }
  }
  for (; i < nvec; i += VER_THREADS) {
    const uint4 v = ldg_stream(rv + i);
    float x[VEC];
#pragma unroll
    for (int j = 0; j < VEC; ++j) x[j] = E::get(v, j);
    consume(x, VEC);
  }
  const int tail = nvec * VEC + tid;
  if (tail < V) {
    float x[1] = {E::load(row, tail)};
    consume(x, 1);
  }
  // block max
  float m = m_run;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
  if (lane == 0) s.red_m[warp] = m;
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < VER_WARPS; ++w) M = fmaxf(M, s.red_m[w]);
  float part = (m_run == -INFINITY) ? 0.0f : s_run * exp2f((m_run - M) * c);
  part = warp_sum(part);
  if (lane == 0) s.red_s[warp] = part;
  __syncthreads();
  if (tid == 0) {
    double z = 0.0;
    for (int w = 0; w < VER_WARPS; ++w) z += s.red_s[w];
    s.M = M;
    s.Zp = z;
  }
  __syncthreads();
}

// Bonus token: first token v in id order with target < sum_{v' <= v} w(v'),
// w = p except at the id-sorted corrections.  Result in s.bonus.  Per chunk
// of VER_THREADS * VEC tokens: float32 per-thread sums and scans, relative to
// the chunk start (the target is rebased per chunk in float64 by thread 0).
template <typename T>
__device__ void bonus_scan(VerShared& s, const uint8_t* row, int V, float c, double target, uint32_t* margins) {
  using E = VElem<T>;
  constexpr int VEC = E::VEC;
  constexpr int CH = VER_THREADS * VEC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float M = s.M;
  const float invZ = static_cast<float>(1.0 / s.Zp);
  const int ncorr = s.ncorr;
  const int nvec_full = static_cast<int>((static_cast<int64_t>(V) * E::ES) / 16);
  int last_pos = -1;
  if (tid == 0) {
    s.bonus = -1;
    s.bonus_last = -1;
    s.running = 0.0;
    s.target_rel = static_cast<float>(target);
  }
  __syncthreads();
  for (int base = 0; base < V; base += CH) {
    const int v0 = base + tid * VEC;
    float w[VEC];
    if (v0 / VEC < nvec_full) {
      const uint4 v = ldg_stream(row + static_cast<int64_t>(v0) * E::ES);
#pragma unroll
      for (int j = 0; j < VEC; ++j) w[j] = E::get(v, j);
    } else {
#pragma unroll
      for (int j = 0; j < VEC; ++j) w[j] = (v0 + j < V) ? E::load(row, v0 + j) : -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < VEC; ++j) w[j] = (w[j] == -INFINITY) ? 0.0f : exp2f((w[j] - M) * c) * invZ;
    // patch corrected tokens in [v0, v0 + VEC)
    if (ncorr > 0 && v0 < V) {
      int lo = 0, hi = ncorr;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s.corr_id[mid] < v0) lo = mid + 1;
        else hi = mid;
      }
      for (int k = lo; k < ncorr && s.corr_id[k] < v0 + VEC; ++k) {
        const int j = s.corr_id[k] - v0;
#pragma unroll
        for (int jj = 0; jj < VEC; ++jj)
          if (jj == j) w[jj] = s.corr_w[k];
      }
    }
    float ts = 0.0f;
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
      ts += w[j];
      if (w[j] > 0.0f && v0 + j < V) last_pos = v0 + j;
    }
    float incl = ts;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s.scan_w[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const float x = s.scan_w[lane];
      float wi = x;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(FULL, wi, o);
        if (lane >= o) wi += t;
      }
      s.scan_x[lane] = wi - x;
      if (lane == 31) s.chunk_total = wi;
    }
    __syncthreads();
    const float before = s.scan_x[warp] + (incl - ts);
    const float after = before + ts;
    const float tr = s.target_rel;
    if (before <= tr && tr < after) {
      // the thread intervals [before, after) are disjoint: at most one thread gets here
      float acc = before;
      int pick = -1, last = -1;
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        if (pick < 0) {
          if (w[j] > 0.0f) last = v0 + j;
          const float nx = acc + w[j];
          if (tr < nx) {
            pick = v0 + j;
            if (margins && (tr - acc < MASS_MARGIN || nx - tr < MASS_MARGIN)) atomicAdd(margins + 1, 1u);
          }
          acc = nx;
        }
      }
      s.bonus = pick >= 0 ? pick : last;
    }
    __syncthreads();
    if (s.bonus >= 0) break;
    if (tid == 0) {
      s.running += s.chunk_total;
      s.target_rel = static_cast<float>(target - s.running);
    }
    __syncthreads();
  }
  if (s.bonus < 0) atomicMax(&s.bonus_last, last_pos);
  __syncthreads();
  if (tid == 0 && s.bonus < 0) s.bonus = s.bonus_last;
  __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(VER_THREADS, 1) verify_kernel(VerifyLaunch L) {
  using E = VElem<T>;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  VerShared& s = *reinterpret_cast<VerShared*>(smem_raw);
  const int b = blockIdx.x, tid = threadIdx.x;
  const spec_tree_t& t = L.tree;
  const int m = L.p.m, D = L.p.depth, K = L.p.K, S = L.S;
  const float Tmp = L.p.temperature;
  const float c = LOG2E / Tmp;
  const int64_t nb = static_cast<int64_t>(b) * t.max_nodes;
  const int n_nodes = t.n_nodes[b];
  for (int i = tid; i < n_nodes; i += VER_THREADS) s.node_parent[i] = t.node_parent[nb + i];
  const int64_t row_bytes = L.row_stride * E::ES;
  const uint8_t* tgt = static_cast<const uint8_t*>(L.target);
  bool nonfinite = false;
  int node = 0, level = 0;
  __syncthreads();
  while (true) {
    const uint8_t* row = tgt + (nb + node) * row_bytes;
    row_stats<T>(s, row, L.V, c, nonfinite);
    // children of the node, verification order: probe first, then by slot
    if (tid == 0) s.nkids = 0;
    __syncthreads();
    for (int i = tid + 1; i < n_nodes; i += VER_THREADS)
      if (s.node_parent[i] == node) {
        const int k = atomicAdd(&s.nkids, 1);
        if (k < SPEC_TREE_MAX_SUPPORT) s.kids[k] = i;
      }
    __syncthreads();
    // a node at depth D is a leaf (also bounds the walk for malformed trees)
    const int nk = level >= D ? 0 : min(s.nkids, SPEC_TREE_MAX_SUPPORT);
    if (tid == 0) {
      // insertion sort: probe first, then slot ascending
      for (int i = 1; i < nk; ++i) {
        const int x = s.kids[i];
        const int kx = t.node_kind[nb + x] == SPEC_TREE_PROBE ? -1 : t.node_slot[nb + x];
        int j = i - 1;
        while (j >= 0) {
          const int y = s.kids[j];
          const int ky = t.node_kind[nb + y] == SPEC_TREE_PROBE ? -1 : t.node_slot[nb + y];
          if (ky <= kx) break;
          s.kids[j + 1] = y;
          --j;
        }
        s.kids[j + 1] = x;
      }
      s.accepted = -1;
      s.residual = 0;
      s.ncorr = 0;
      s.Zr = 1.0;
    }
    __syncthreads();
    const float M = s.M;
    const float invZp = static_cast<float>(1.0 / s.Zp);
    int64_t srow = -1;
    if (nk > 0) {
      srow = static_cast<int64_t>(b) * t.n_rows + t.node_exp_row[nb + node];
      const float zT = t.sup_zT[srow];
      if (tid < S) {
        const int v = t.sup_id[srow * t.sup_stride + tid];
        const float x = E::load(row, v);
        const float p = expf((x - M) / Tmp) * invZp;
        s.p_sup[tid] = p;
        const float qt = (tid >= m && zT > 0.0f) ? t.sup_qT[srow * t.sup_stride + tid] / zT : 0.0f;
        s.qt_sup[tid] = qt;
        s.w_sup[tid] = p;
      }
      __syncthreads();
      if (tid == 0) {
        const float* uv = L.u_verify + (static_cast<int64_t>(b) * D + level) * K;
        const int pp = t.probe_pos[srow];
        int j = 0, i0 = 0;
        double Zr = 1.0;
        auto rank_of = [&](int node_i) -> int {
          const int kind = t.node_kind[nb + node_i], slot = t.node_slot[nb + node_i];
          if (kind == SPEC_TREE_DET) return slot;
          if (kind == SPEC_TREE_PROBE) return pp;
          int r = m + slot - m - (pp >= 0 ? 1 : 0);
          if (pp >= 0 && r >= pp) ++r;
          return r;
        };
        if (nk > 0 && t.node_kind[nb + s.kids[0]] == SPEC_TREE_PROBE) {
          const int r = pp;
          const double p = s.p_sup[r], qt = s.qt_sup[r];
          const float u = uv[0];
          if (L.margins && fabs(u * qt - p) < MASS_MARGIN) atomicAdd(L.margins, 1u);
          if (static_cast<double>(u) * qt < p) {
            s.accepted = s.kids[0];
          } else {
            // residual max(0, p - q~) on the tail, mass 1 - sum_tail min(p, q~)
            double smin = 0.0;
            for (int k = m; k < S; ++k) {
              const float pk = s.p_sup[k], qk = s.qt_sup[k];
              smin += fminf(pk, qk);
              s.w_sup[k] = fmaxf(0.0f, pk - qk);
            }
            Zr = 1.0 - smin;
            s.residual = 1;
            j = 1;
          }
          i0 = 1;
        }
        if (s.accepted < 0) {
          bool empty = false;
          for (int i = i0; i < nk; ++i, ++j) {
            if (Zr <= 0.0) {
              empty = true;
              break;
            }
            const int r = rank_of(s.kids[i]);
            const double w = s.w_sup[r];
            const float u = uv[j];
            if (L.margins && fabs(u * Zr - w) < MASS_MARGIN) atomicAdd(L.margins, 1u);
            if (static_cast<double>(u) * Zr < w) {
              s.accepted = s.kids[i];
              break;
            }
            Zr -= w;
            s.w_sup[r] = 0.0f;
          }
          if (s.accepted < 0 && !empty && Zr <= 0.0) empty = true;
          if (empty) {
            // rounding emptied the residual: bonus from p
            set_status(L.status, SPEC_TREE_S_RESIDUAL_EMPTY);
            for (int k = 0; k < S; ++k) s.w_sup[k] = s.p_sup[k];
            s.residual = 0;
            Zr = 1.0;
          }
        }
        s.Zr = Zr;
      }
      __syncthreads();
    }
    const int acc = s.accepted;
    if (acc >= 0) {
      if (tid == 0) {
        L.out_tok[static_cast<int64_t>(b) * (D + 1) + level] = t.node_token[nb + acc];
        L.out_node[static_cast<int64_t>(b) * (D + 1) + level] = acc;
      }
      node = acc;
      ++level;
      __syncthreads();
      continue;
    }
    // bonus: corrections are the support tokens whose w differs from p
    if (nk > 0) {
      if (tid < S) {
        const bool corr = s.w_sup[tid] != s.p_sup[tid];
        const int v = t.sup_id[srow * t.sup_stride + tid];
        if (corr) {
          int r = 0;
          for (int k = 0; k < S; ++k) {
            const bool ck = s.w_sup[k] != s.p_sup[k];
            if (ck && t.sup_id[srow * t.sup_stride + k] < v) ++r;
          }
          s.corr_id[r] = v;
          s.corr_w[r] = s.w_sup[tid];
          atomicAdd(&s.ncorr, 1);
        }
      }
      __syncthreads();
    }
    const double target = static_cast<double>(L.u_bonus[b]) * s.Zr;
    bonus_scan<T>(s, row, L.V, c, target, L.margins);
    if (tid == 0) {
      int32_t* ot = L.out_tok + static_cast<int64_t>(b) * (D + 1);
      int32_t* on = L.out_node + static_cast<int64_t>(b) * (D + 1);
      ot[level] = s.bonus;
      on[level] = -1;
      for (int k = level + 1; k <= D; ++k) {
        ot[k] = -1;
        on[k] = -1;
      }
      L.accept_len[b] = level;
    }
    break;
  }
  if (nonfinite) set_status(L.status, SPEC_TREE_S_NONFINITE_TARGET);
}

cudaError_t launch_verify(const VerifyLaunch& L, cudaStream_t stream) {
  if (L.B == 0) return cudaSuccess;
  const int smem = static_cast<int>(sizeof(VerShared));
  if (L.dtype == SPEC_TREE_BF16) {
    cudaError_t err =
        cudaFuncSetAttribute(verify_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    verify_kernel<__nv_bfloat16><<<L.B, VER_THREADS, smem, stream>>>(L);
  } else {
    cudaError_t err = cudaFuncSetAttribute(verify_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    verify_kernel<float><<<L.B, VER_THREADS, smem, stream>>>(L);
  }
  return cudaGetLastError();
}

}  // namespace st
