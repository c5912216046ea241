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
// Per level the CTA streams the node's target row once with 16-byte loads;
// warp w owns a contiguous slice of the row and keeps the slice's maximum and
// sum of exp2((t - max) * log2(e) / T), so the row normaliser and the mass of
// every slice come out of the same pass.  The <= |S| support tokens of the
// node's draft row (the tail and the children) are gathered for exact p, the
// residual is formed in parallel, and thread 0 takes the <= K decisions.  For
// the bonus token the slice masses locate the slice that holds it, and only
// that slice is read again and scanned in token-id order.
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
  int32_t kid_by_slot[SPEC_TREE_MAX_SUPPORT];  // child node of each sibling slot, -1 if pruned
  float p_sup[SPEC_TREE_MAX_SUPPORT];          // p at support ranks of the node's draft row
  float w_sup[SPEC_TREE_MAX_SUPPORT];          // residual at support ranks
  float slice_m[VER_WARPS];                    // slice maximum (logit)
  float slice_s[VER_WARPS];                    // slice sum of exp2((t - slice_m) * c)
  float slice_corr[VER_WARPS];                 // per slice: sum over corrected tokens of (p - w)
  float red[VER_WARPS];
  int32_t corr_tok[SPEC_TREE_MAX_SUPPORT];     // corrected tokens inside the bonus slice
  float corr_w[SPEC_TREE_MAX_SUPPORT];
  float scan_w[VER_WARPS];
  int ncorr;
  float M;       // row maximum
  double Zp;     // row sum of exp2((t - M) * c)
  double Zr;     // residual mass
  int accepted;  // accepted child node or -1
  int bonus;
  int bonus_last;
  int bonus_slice;
  float bonus_target;  // target mass relative to the start of the bonus slice
};

// 2^x on the special-function unit (PTX ex2.approx.ftz: a few ulp; results
// below 2^-126 flush to zero, which changes a row sum by at most 2^-126).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T>
struct VElem;
template <>
struct VElem<__nv_bfloat16> {
  static constexpr int VEC = 8, ES = 2;
  __device__ static float get(const uint4& v, int j) {
    const uint32_t w = (j < 2) ? v.x : (j < 4) ? v.y : (j < 6) ? v.z : v.w;
    return __uint_as_float((j & 1) ? (w & 0xffff0000u) : (w << 16));
  }
  __device__ static float load(const uint8_t* row, int v) {
    return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(row)[v]) << 16);
  }
  // maximum of the 8 elements, NaN-propagating
  __device__ static float vmax(const uint4& v) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&v.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&v.w);
    const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    return __bfloat162float(__hmax_nan(m.x, m.y));
  }
};
template <>
struct VElem<float> {
  static constexpr int VEC = 4, ES = 4;
  __device__ static float get(const uint4& v, int j) {
    return __uint_as_float((j == 0) ? v.x : (j == 1) ? v.y : (j == 2) ? v.z : v.w);
  }
  __device__ static float load(const uint8_t* row, int v) { return reinterpret_cast<const float*>(row)[v]; }
  __device__ static float vmax(const uint4& v) {
    const float a = __uint_as_float(v.x), b = __uint_as_float(v.y), c = __uint_as_float(v.z),
                d = __uint_as_float(v.w);
    const float m = fmaxf(fmaxf(a, b), fmaxf(c, d));
    return (a != a || b != b || c != c || d != d) ? __int_as_float(0x7fffffff) : m;
  }
};

// Slice of warp w: vectors [w * per, min((w + 1) * per, nvec)); the scalar
// tail (V not a multiple of the vector width) belongs to the last warp.
struct Slice {
  int v0, v1;
  __device__ Slice(int w, int nvec) {
    const int per = (nvec + VER_WARPS - 1) / VER_WARPS;
    v0 = min(w * per, nvec);
    v1 = min(v0 + per, nvec);
  }
};

__device__ __forceinline__ int slice_of_token(int v, int nvec, int vec) {
  const int per = (nvec + VER_WARPS - 1) / VER_WARPS;
  if (v >= nvec * vec || per == 0) return VER_WARPS - 1;
  return min((v / vec) / per, VER_WARPS - 1);
}

// Row statistics: per-slice maximum and sum of exp2((t - m) * c), the row
// maximum M and Zp = sum exp2((t - M) * c), c = log2(e) / T.  Per lane:
// online maximum with rescaling, compensated float32 sums of 8-element vector
// sums; lanes combine in float32, slices in float64.
template <typename T>
__device__ void row_stats(VerShared& s, const uint8_t* row, int V, float c, bool& nonfinite) {
  using E = VElem<T>;
  constexpr int VEC = E::VEC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nvec = static_cast<int>((static_cast<int64_t>(V) * E::ES) / 16);
  const Slice sl(warp, nvec);
  float m_run = -INFINITY, s_run = 0.0f, comp = 0.0f;
  auto rescale = [&](float vm) {
    const float f = ex2((m_run - vm) * c);
    s_run *= f;
    comp *= f;
    m_run = vm;
  };
  auto consume = [&](const uint4& v) {
    const float vm = E::vmax(v);
    if (!(vm < INFINITY)) {  // NaN or +inf in the row
      nonfinite = true;
      return;
    }
    if (vm == -INFINITY) return;
    if (vm > m_run) rescale(vm);
    float vs = 0.0f;
#pragma unroll
    for (int j = 0; j < VEC; ++j) vs += ex2((E::get(v, j) - m_run) * c);
    const float y = vs - comp;
    const float t = s_run + y;
    comp = (t - s_run) - y;
    s_run = t;
  };
  const uint4* rv = reinterpret_cast<const uint4*>(row);
  int i = sl.v0 + lane;
  for (; i + 96 < sl.v1; i += 128) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = ldg_stream(rv + i + 32 * u);
#pragma unroll
    for (int u = 0; u < 4; ++u) consume(v[u]);
  }
  for (; i < sl.v1; i += 32) consume(ldg_stream(rv + i));
  if (warp == VER_WARPS - 1) {
    const int tk = nvec * VEC + lane;
    if (tk < V) {
      const float x = E::load(row, tk);
      if (!(x < INFINITY)) nonfinite = true;
      if (x > -INFINITY && x < INFINITY) {
        if (x > m_run) rescale(x);
        s_run += ex2((x - m_run) * c);
      }
    }
  }
  // combine lanes: slice maximum and sum relative to it
  float m = m_run;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
  float part = (m_run == -INFINITY) ? 0.0f : (s_run - comp) * ex2((m_run - m) * c);
  part = warp_sum(part);
  if (lane == 0) {
    s.slice_m[warp] = m;
    s.slice_s[warp] = part;
  }
  __syncthreads();
  if (tid == 0) {
    float M = -INFINITY;
    for (int w = 0; w < VER_WARPS; ++w) M = fmaxf(M, s.slice_m[w]);
    double z = 0.0;
    for (int w = 0; w < VER_WARPS; ++w)
      if (s.slice_m[w] > -INFINITY) z += static_cast<double>(s.slice_s[w]) * ex2((s.slice_m[w] - M) * c);
    s.M = M;
    s.Zp = z;
  }
  __syncthreads();
}

// Support rank of the child in sibling slot `slot` (DET 0..m-1 -> ranks
// 0..m-1, PROBE m -> the probe's rank, FILL -> next tail ranks skipping the probe).
__device__ __forceinline__ int rank_of_slot(int slot, int m, int pp) {
  if (slot < m) return slot;
  if (slot == m && pp >= 0) return pp;
  int r = slot - (pp >= 0 ? 1 : 0);
  if (pp >= 0 && r >= pp) ++r;
  return r;
}

template <typename T>
__global__ void __launch_bounds__(VER_THREADS, 1) verify_kernel(VerifyLaunch L) {
  using E = VElem<T>;
  constexpr int VEC = E::VEC;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  VerShared& s = *reinterpret_cast<VerShared*>(smem_raw);
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const spec_tree_t& t = L.tree;
  const int m = L.p.m, D = L.p.depth, K = L.p.K, S = L.S, V = L.V;
  const float Tmp = L.p.temperature;
  const float c = LOG2E / Tmp;
  const int64_t nb = static_cast<int64_t>(b) * t.max_nodes;
  const int n_nodes = min(t.n_nodes[b], t.max_nodes);
  for (int i = tid; i < n_nodes; i += VER_THREADS) s.node_parent[i] = t.node_parent[nb + i];
  const int64_t row_bytes = L.row_stride * E::ES;
  const uint8_t* tgt = static_cast<const uint8_t*>(L.target);
  const int nvec = static_cast<int>((static_cast<int64_t>(V) * E::ES) / 16);
  bool nonfinite = false;
  int node = 0, level = 0;
  int32_t* ot = L.out_tok + static_cast<int64_t>(b) * (D + 1);
  int32_t* on = L.out_node + static_cast<int64_t>(b) * (D + 1);
  __syncthreads();
  while (true) {
    const uint8_t* row = tgt + (nb + node) * row_bytes;
    if (tid < K) s.kid_by_slot[tid] = -1;
    if (tid == 0) {
      s.accepted = -1;
      s.Zr = 1.0;
      s.ncorr = 0;
    }
    row_stats<T>(s, row, V, c, nonfinite);
    // children of the node by sibling slot; a node at depth D is a leaf
    // (which also bounds the walk for malformed trees)
    int nk = 0;
    if (level < D) {
      for (int i = tid + 1; i < n_nodes; i += VER_THREADS)
        if (s.node_parent[i] == node) {
          const int slot = t.node_slot[nb + i];
          if (slot >= 0 && slot < K) s.kid_by_slot[slot] = i;
        }
      __syncthreads();
      for (int k = 0; k < K; ++k) nk += s.kid_by_slot[k] >= 0;
    }
    const float M = s.M;
    const float invZp = static_cast<float>(1.0 / s.Zp);
    int64_t srow = -1;
    if (nk > 0) {
      srow = static_cast<int64_t>(b) * t.n_rows + t.node_exp_row[nb + node];
      const int pp = t.probe_pos[srow];
      const int probe_node = (pp >= 0) ? s.kid_by_slot[m] : -1;
      const bool residual = probe_node >= 0;  // the tail residual applies iff the probe child survived
      const float zT = t.sup_zT[srow];
      float mn = 0.0f;
      if (tid < S) {
        const int v = t.sup_id[srow * t.sup_stride + tid];
        const float p = expf((E::load(row, v) - M) / Tmp) * invZp;
        const float qt = (tid >= m && zT > 0.0f) ? t.sup_qT[srow * t.sup_stride + tid] / zT : 0.0f;
        s.p_sup[tid] = p;
        s.w_sup[tid] = (residual && tid >= m) ? fmaxf(0.0f, p - qt) : p;
        mn = (residual && tid >= m) ? fminf(p, qt) : 0.0f;
      }
      mn = warp_sum(mn);
      if (lane == 0) s.red[warp] = mn;
      __syncthreads();
      if (tid == 0) {
        const float* uv = L.u_verify + (static_cast<int64_t>(b) * D + level) * K;
        int j = 0;
        double Zr = 1.0;
        bool empty = false;
        if (probe_node >= 0) {
          const double p = s.p_sup[pp];
          const double qt = static_cast<double>(t.sup_qT[srow * t.sup_stride + pp]) / zT;
          const float u = uv[0];
          if (L.margins && fabs(u * qt - p) < MASS_MARGIN) atomicAdd(L.margins, 1u);
          if (static_cast<double>(u) * qt < p) {
            s.accepted = probe_node;
          } else {
            double smin = 0.0;
            for (int w = 0; w < (S + 31) / 32; ++w) smin += s.red[w];
            Zr = 1.0 - smin;
            j = 1;
          }
        }
        if (s.accepted < 0) {
          for (int slot = 0; slot < K; ++slot) {
            const int kid = s.kid_by_slot[slot];
            if (kid < 0 || kid == probe_node) continue;
            if (Zr <= 0.0) {
              empty = true;
              break;
            }
            const int r = rank_of_slot(slot, m, pp);
            const double w = s.w_sup[r];
            const float u = uv[j];
            if (L.margins && fabs(u * Zr - w) < MASS_MARGIN) atomicAdd(L.margins, 1u);
            if (static_cast<double>(u) * Zr < w) {
              s.accepted = kid;
              break;
            }
            Zr -= w;
            s.w_sup[r] = 0.0f;
            ++j;
          }
          if (s.accepted < 0 && !empty && Zr <= 0.0) empty = true;
          if (empty) {
            // rounding emptied the residual: the bonus is drawn from p
            set_status(L.status, SPEC_TREE_S_RESIDUAL_EMPTY);
            for (int k = 0; k < S; ++k) s.w_sup[k] = s.p_sup[k];
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
        ot[level] = t.node_token[nb + acc];
        on[level] = acc;
      }
      node = acc;
      ++level;
      __syncthreads();
      continue;
    }
    // ------------------------------------------------------------- bonus ---
    // w = p except at support tokens whose residual differs; slice masses of w
    if (tid < VER_WARPS) s.slice_corr[tid] = 0.0f;
    __syncthreads();
    if (nk > 0 && tid < S) {
      const float d = s.p_sup[tid] - s.w_sup[tid];
      if (d != 0.0f)
        atomicAdd(&s.slice_corr[slice_of_token(t.sup_id[srow * t.sup_stride + tid], nvec, VEC)], d);
    }
    __syncthreads();
    if (tid == 0) {
      const double target = static_cast<double>(L.u_bonus[b]) * s.Zr;
      double acc_mass = 0.0, before = 0.0, before_last = 0.0;
      int pick = -1, last = -1;
      for (int w = 0; w < VER_WARPS; ++w) {
        double mass = s.slice_m[w] > -INFINITY
                          ? static_cast<double>(s.slice_s[w]) * ex2((s.slice_m[w] - M) * c) / s.Zp
                          : 0.0;
        mass -= s.slice_corr[w];
        if (mass > 0.0) {
          last = w;
          before_last = acc_mass;
        }
        if (pick < 0 && mass > 0.0 && target < acc_mass + mass) {
          pick = w;
          before = acc_mass;
        }
        acc_mass += mass;
      }
      if (pick < 0) {  // rounding left the target past the total: the last slice with mass
        pick = last < 0 ? VER_WARPS - 1 : last;
        before = before_last;
      }
      s.bonus_slice = pick;
      s.bonus_target = static_cast<float>(target - before);
      s.bonus = -1;
      s.bonus_last = -1;
    }
    __syncthreads();
    const int bs = s.bonus_slice;
    const Slice sl(bs, nvec);
    const int t0 = sl.v0 * VEC;
    const int t1 = (bs == VER_WARPS - 1) ? V : sl.v1 * VEC;
    // corrected tokens inside the slice
    if (nk > 0 && tid < S) {
      const float wv = s.w_sup[tid];
      if (wv != s.p_sup[tid]) {
        const int v = t.sup_id[srow * t.sup_stride + tid];
        if (v >= t0 && v < t1) {
          const int k = atomicAdd(&s.ncorr, 1);
          s.corr_tok[k] = v;
          s.corr_w[k] = wv;
        }
      }
    }
    __syncthreads();
    // scan the slice in id order: thread i handles tokens [base + VEC * i, + VEC)
    {
      const int ncorr = s.ncorr;
      const float invZ = static_cast<float>(1.0 / s.Zp);
      const float tr = s.bonus_target;
      float base_run = 0.0f;
      int last_pos = -1;
      for (int cb = t0; cb < t1; cb += VER_THREADS * VEC) {
        const int v0 = cb + tid * VEC;
        float w[VEC];
        if (v0 + VEC <= t1 && v0 / VEC < nvec) {
          const uint4 v = ldg_stream(row + static_cast<int64_t>(v0) * E::ES);
#pragma unroll
          for (int j = 0; j < VEC; ++j) w[j] = E::get(v, j);
        } else {
#pragma unroll
          for (int j = 0; j < VEC; ++j) w[j] = (v0 + j < t1) ? E::load(row, v0 + j) : -INFINITY;
        }
        float ts = 0.0f;
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
          w[j] = (w[j] == -INFINITY) ? 0.0f : ex2((w[j] - M) * c) * invZ;
          for (int k = 0; k < ncorr; ++k)
            if (s.corr_tok[k] == v0 + j) w[j] = s.corr_w[k];
          ts += w[j];
          if (w[j] > 0.0f) last_pos = v0 + j;
        }
        float incl = ts;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float x = __shfl_up_sync(FULL, incl, o);
          if (lane >= o) incl += x;
        }
        if (lane == 31) s.scan_w[warp] = incl;
        __syncthreads();
        float wbefore = 0.0f, total = 0.0f;
        for (int k = 0; k < VER_WARPS; ++k) {
          const float x = s.scan_w[k];
          if (k < warp) wbefore += x;
          total += x;
        }
        const float before = base_run + wbefore + incl - ts;
        if (ts > 0.0f && before <= tr && tr < before + ts) {
          // the thread intervals [before, before + ts) are disjoint: one thread at most
          float acc = before;
          int pick = -1, lastp = -1;
#pragma unroll
          for (int j = 0; j < VEC; ++j) {
            if (pick < 0) {
              if (w[j] > 0.0f) lastp = v0 + j;
              const float nx = acc + w[j];
              if (tr < nx) {
                pick = v0 + j;
                if (L.margins && (tr - acc < MASS_MARGIN || nx - tr < MASS_MARGIN)) atomicAdd(L.margins + 1, 1u);
              }
              acc = nx;
            }
          }
          s.bonus = pick >= 0 ? pick : lastp;
        }
        base_run += total;
        __syncthreads();
        if (s.bonus >= 0) break;
      }
      if (s.bonus < 0 && last_pos >= 0) atomicMax(&s.bonus_last, last_pos);
      __syncthreads();
    }
    if (tid == 0) {
      int bonus = s.bonus;
      if (bonus < 0) bonus = s.bonus_last;
      if (bonus < 0) bonus = t1 - 1;
      ot[level] = bonus;
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
