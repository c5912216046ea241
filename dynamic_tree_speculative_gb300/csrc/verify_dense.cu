// Verification of trees built on a dense draft support (|S| = V above
// SPEC_TREE_MAX_SUPPORT tokens), sm_103a.
//
// RheoSampling notes, Method / Key design 3 (optimal-transport verification)
// with the renormalised tail law over the whole vocabulary:
// q~_T(v) = q_T(v) / z_T for every token v but the m deterministic ones.  Only
// the support's first ranks and the probe are stored, so q_T(v) is recomputed
// from the node's draft row d: q_T(v) = exp((d_v - d_max) / T) * q_T(x_1), with
// d_max the rank-0 logit and q_T(x_1) = 1 / sum exp((d - d_max) / T) as the
// build wrote it.
//
// One CTA of VD_THREADS threads per tree, plain 16-byte loads.  Per level:
//   1. the target row's maximum M and Zp = sum exp((t - M) / T) (online per
//      thread, combined across the block);
//   2. thread 0 takes the accept tests in verification order with the level's
//      uniforms: the probe with u < p / q~, a one-hot child with u < w / Zr;
//   3. once the probe is tested and rejected, one pass over the target and
//      draft rows gives sum_tail min(a, c q~) (a = p with the rejected one-hot
//      children zeroed; c = 1 probe first, c = Zr probe last), so the residual
//      w = max(0, a - c q~) on the tail has mass Zr - that sum;
//   4. when every child is rejected, or the node has none, the bonus is the
//      first token in id order whose cumulative w exceeds u_bonus * Zr: a scan
//      in rounds of VD_THREADS consecutive vectors, each with a block scan in
//      float32 and the carry of the earlier rounds in float64 (the GPU's
//      float64 rate is a small fraction of its float32 rate: with every
//      partial sum in float64 the scan took most of the kernel).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "st_common.cuh"
#include "st_kernels.h"

namespace st {
namespace {

constexpr int VD_THREADS = 1024;
constexpr int VD_WARPS = VD_THREADS / 32;
constexpr int VD_MAX_K = SPEC_TREE_DENSE_MAX_K;
constexpr float VD_LOG2E = 1.4426950408889634f;
constexpr float VD_MARGIN = 1e-6f;

template <typename T>
struct VDElem;
template <>
struct VDElem<__nv_bfloat16> {
  static constexpr int VEC = 8;
  static constexpr int ES = 2;
  __device__ static float get(const uint4& v, int j) {
    const uint32_t w = (j < 2) ? v.x : (j < 4) ? v.y : (j < 6) ? v.z : v.w;
    return __uint_as_float(((w >> (16 * (j & 1))) & 0xffffu) << 16);
  }
  __device__ static float load(const uint8_t* row, int i) {
    return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(row)[i]) << 16);
  }
};
template <>
struct VDElem<float> {
  static constexpr int VEC = 4;
  static constexpr int ES = 4;
  __device__ static float get(const uint4& v, int j) {
    return __uint_as_float(j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w);
  }
  __device__ static float load(const uint8_t* row, int i) { return reinterpret_cast<const float*>(row)[i]; }
};

struct VDShared {
  int32_t nd_parent[SPEC_TREE_MAX_NODES];
  int32_t nd_slot[SPEC_TREE_MAX_NODES];
  int32_t nd_kind[SPEC_TREE_MAX_NODES];
  int32_t nd_tok[SPEC_TREE_MAX_NODES];
  int32_t nd_exp[SPEC_TREE_MAX_NODES];
  int kid[VD_MAX_K];     // node index of the child in each slot, -1 if none
  int ktok[VD_MAX_K];    // its token and kind
  int kkind[VD_MAX_K];
  float kp[VD_MAX_K];    // p of the child's token
  float kq[VD_MAX_K];    // q~_T of the child's token (0 for DET children)
  float uv[VD_MAX_K];    // the level's accept uniforms
  int det[VD_MAX_K];     // the node's DET tokens (support ranks 0..m-1)
  int zero[VD_MAX_K];    // rejected one-hot children (w = 0)
  int nzero;
  float red_m[VD_WARPS];
  float red_s[VD_WARPS];
  int flag;
  // broadcast state of the level
  float M, invZp, c;  // target normaliser; c = log2(e) / T
  float dmax, qscale;  // draft rank-0 logit; q_T(x_1) / z_T
  float cres;          // residual scale c (probe first 1, probe last Zr before the probe)
  int residual;        // the residual applies on the tail
  int need_pass;       // 0: none, 1: residual mass before the one-hot children, 2: after (probe last)
  int accepted;
  int empty;
  float Zr;
  int j;               // next decision index of the level
  int bonus, bonus_last;
  double bonus_target;
};

// Calls f(id, t, d) for every element of thread tid's vectors tid, tid + VD_THREADS, ...
// and the scalar tail; d (the draft logit) is only loaded when `with_draft`.
template <typename T, typename F>
__device__ __forceinline__ void for_rows(const uint8_t* trow, const uint8_t* drow, int V, int nvec, bool with_draft,
                                         F f) {
  using E = VDElem<T>;
  const int tid = threadIdx.x;
  for (int vi = tid; vi < nvec; vi += VD_THREADS) {
    const uint4 tv = ldg_stream(trow + static_cast<int64_t>(vi) * 16);
    uint4 dv = make_uint4(0, 0, 0, 0);
    if (with_draft) dv = ldg_stream(drow + static_cast<int64_t>(vi) * 16);
#pragma unroll
    for (int j = 0; j < E::VEC; ++j) f(vi * E::VEC + j, E::get(tv, j), with_draft ? E::get(dv, j) : 0.0f);
  }
  const int id = nvec * E::VEC + tid;
  if (id < V) f(id, E::load(trow, id), with_draft ? E::load(drow, id) : 0.0f);
}

// 2^x on the special-function unit (PTX ex2.approx.ftz: a few ulp; results
// below 2^-126 flush to zero).  Every exponential of the kernel uses it, so
// the children's p and q~ and the row passes agree.
__device__ __forceinline__ float vd_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ bool in_list(const int* list, int n, int v) {
  for (int k = 0; k < n; ++k)
    if (list[k] == v) return true;
  return false;
}

template <typename T>
__global__ void __launch_bounds__(VD_THREADS, 1) verify_dense_kernel(VerifyLaunch L) {
  using E = VDElem<T>;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  VDShared& s = *reinterpret_cast<VDShared*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const spec_tree_t& t = L.tree;
  const int K = L.p.K, m = L.p.m, D = L.p.depth, V = L.V;
  const int es = E::ES;
  const int nvec = static_cast<int>((static_cast<int64_t>(V) * es) / 16);
  const bool probe_first = L.p.verify_order == SPEC_TREE_PROBE_FIRST;
  const float c = L.p.temperature == 1.0f ? VD_LOG2E : VD_LOG2E / L.p.temperature;
  grid_dependency_wait();
  grid_dependents_launch();

  const int64_t nb = static_cast<int64_t>(b) * t.max_nodes;
  const int nn = min(t.n_nodes[b], t.max_nodes);
  for (int i = tid; i < nn; i += VD_THREADS) {
    s.nd_parent[i] = t.node_parent[nb + i];
    s.nd_slot[i] = t.node_slot[nb + i];
    s.nd_kind[i] = t.node_kind[nb + i];
    s.nd_tok[i] = t.node_token[nb + i];
    s.nd_exp[i] = t.node_exp_row[nb + i];
  }
  __syncthreads();
  int32_t* ot = L.out_tok + static_cast<int64_t>(b) * (D + 1);
  int32_t* on = L.out_node + static_cast<int64_t>(b) * (D + 1);
  bool nonfinite = false;
  int node = 0, level = 0;
  while (true) {
    const uint8_t* trow = static_cast<const uint8_t*>(L.target) + (nb + node) * L.row_stride * es;
    const int er = s.nd_exp[node];
    const bool has_row = er >= 0 && er < t.n_rows && level < D;
    const int64_t srow = static_cast<int64_t>(b) * t.n_rows + (has_row ? er : 0);
    const uint8_t* drow = static_cast<const uint8_t*>(L.draft) + srow * L.draft_row_stride * es;
    if (tid < K) {
      s.kid[tid] = -1;
      s.uv[tid] = level < D ? L.u_verify[(static_cast<int64_t>(b) * D + level) * K + tid] : 0.0f;
    }
    if (tid == 0) {
      s.nzero = 0;
      s.need_pass = 0;
      s.residual = 0;
      s.accepted = -1;
      s.empty = 0;
      s.Zr = 1.0f;
      s.j = 0;
      s.cres = 1.0f;
    }
    __syncthreads();
    if (has_row)
      for (int i = tid + 1; i < nn; i += VD_THREADS)
        if (s.nd_parent[i] == node && s.nd_slot[i] >= 0 && s.nd_slot[i] < K) s.kid[s.nd_slot[i]] = i;

    // 1. the target row's normaliser, online per thread
    float mx = -INFINITY, sm = 0.0f;
    for_rows<T>(trow, trow, V, nvec, false, [&](int, float x, float) {
      if (!(x < INFINITY) && !(x == -INFINITY)) nonfinite = true;  // NaN or +inf
      if (x > mx) {
        sm = sm * vd_ex2((mx - x) * c) + 1.0f;
        mx = x;
      } else if (x > -INFINITY) {
        sm += vd_ex2((x - mx) * c);
      }
    });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float om = __shfl_xor_sync(FULL, mx, o), os = __shfl_xor_sync(FULL, sm, o);
      const float nm = fmaxf(mx, om);
      sm = (mx > -INFINITY ? sm * vd_ex2((mx - nm) * c) : 0.0f) + (om > -INFINITY ? os * vd_ex2((om - nm) * c) : 0.0f);
      mx = nm;
    }
    if (lane == 0) {
      s.red_m[warp] = mx;
      s.red_s[warp] = sm;
    }
    __syncthreads();
    if (tid == 0) {
      float M = -INFINITY;
      for (int w = 0; w < VD_WARPS; ++w) M = fmaxf(M, s.red_m[w]);
      double Z = 0.0;
      for (int w = 0; w < VD_WARPS; ++w)
        if (s.red_m[w] > -INFINITY) Z += static_cast<double>(s.red_s[w]) * vd_ex2((s.red_m[w] - M) * c);
      s.M = M;
      s.invZp = static_cast<float>(1.0 / Z);
    }
    __syncthreads();
    const float M = s.M, invZp = s.invZp;

    // the children's p and q~ (q~ from the draft row), the DET tokens, the draft's rank-0 logit
    if (has_row) {
      const int64_t sb = srow * t.sup_stride;
      if (tid < m && tid < K) s.det[tid] = t.sup_id[sb + tid];
      if (tid == 0) {
        const int top = t.sup_id[sb];
        s.dmax = top >= 0 && top < V ? E::load(drow, top) : 0.0f;
        const float zT = t.sup_zT[srow];
        s.qscale = zT > 0.0f ? t.sup_qT[sb] / zT : 0.0f;
      }
    }
    __syncthreads();
    if (tid < K) {
      const int kd = s.kid[tid];
      if (kd >= 0) {
        const int tok = s.nd_tok[kd];
        const int kind = s.nd_kind[kd];
        s.ktok[tid] = tok;
        s.kkind[tid] = kind;
        const bool ok = tok >= 0 && tok < V;
        s.kp[tid] = ok ? vd_ex2((E::load(trow, tok) - M) * c) * invZp : 0.0f;
        s.kq[tid] = (ok && kind != SPEC_TREE_DET) ? vd_ex2((E::load(drow, tok) - s.dmax) * c) * s.qscale : 0.0f;
      }
    }
    __syncthreads();

    // 2. decisions up to the first full-row pass they need
    const int pslot = (m < K && s.kid[m] >= 0 && s.kkind[m] == SPEC_TREE_PROBE) ? m : -1;
    if (tid == 0) {
      if (pslot >= 0 && probe_first) {
        const float u = s.uv[0], p = s.kp[pslot], q = s.kq[pslot];
        if (L.margins && fabsf(u * q - p) < VD_MARGIN * q) atomicAdd(L.margins, 1u);
        s.j = 1;
        if (u * q < p) {
          s.accepted = s.kid[pslot];
        } else {
          s.need_pass = 1;  // the residual mass of the probe's rejection
          s.residual = 1;
          s.cres = 1.0f;
        }
      }
    }
    __syncthreads();
    for (int phase = 0; phase < 2; ++phase) {
      if (s.need_pass) {
        // 3. sum over the tail of min(a, c q~), a = p with the rejected one-hot children zeroed
        const float cres = s.cres, dmax = s.dmax, qscale = s.qscale;
        const int nz = s.nzero;
        float acc = 0.0f, comp = 0.0f;
        for_rows<T>(trow, drow, V, nvec, true, [&](int id, float x, float dl) {
          if (in_list(s.det, m, id)) return;
          const float a = in_list(s.zero, nz, id) ? 0.0f : vd_ex2((x - M) * c) * invZp;
          const float q = vd_ex2((dl - dmax) * c) * qscale;
          const float y = fminf(a, cres * q) - comp;
          const float tt = acc + y;
          comp = (tt - acc) - y;
          acc = tt;
        });
        // warp sums in float, the 32 of them added in double by thread 0 (the
        // SM's float64 rate is a small fraction of its float32 rate)
        float part = acc - comp;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(FULL, part, o);
        if (lane == 0) s.red_s[warp] = part;
        __syncthreads();
        if (tid == 0) {
          double tot = 0.0;
          for (int w = 0; w < VD_WARPS; ++w) tot += static_cast<double>(s.red_s[w]);
          s.Zr = static_cast<float>(static_cast<double>(s.Zr) - tot);
          s.need_pass = 0;
        }
        __syncthreads();
      }
      if (phase == 1) break;
      if (tid == 0 && s.accepted < 0) {
        float Zr = s.Zr;
        int j = s.j;
        // one-hot children in slot order (the probe first is already decided)
        for (int slot = 0; slot < K && s.accepted < 0; ++slot) {
          if (s.kid[slot] < 0 || slot == pslot) continue;
          if (Zr <= 0.0f) {
            s.empty = 1;
            break;
          }
          const float w = (s.residual && s.kkind[slot] != SPEC_TREE_DET) ? fmaxf(0.0f, s.kp[slot] - s.cres * s.kq[slot])
                                                                         : s.kp[slot];
          const float u = s.uv[j];
          if (L.margins && fabsf(u * Zr - w) < VD_MARGIN * Zr) atomicAdd(L.margins, 1u);
          ++j;
          if (u * Zr < w) {
            s.accepted = s.kid[slot];
            break;
          }
          Zr -= w;
          s.zero[s.nzero++] = s.ktok[slot];
        }
        if (s.accepted < 0 && !s.empty && pslot >= 0 && !probe_first) {
          // the probe last, against the residual the one-hot rejections left
          if (Zr <= 0.0f) {
            s.empty = 1;
          } else {
            const float w = s.kp[pslot], q = s.kq[pslot], u = s.uv[j];
            if (L.margins && fabsf(u * q * Zr - w) < VD_MARGIN * q * Zr) atomicAdd(L.margins, 1u);
            ++j;
            if (u * q * Zr < w) {
              s.accepted = s.kid[pslot];
            } else {
              s.need_pass = 2;
              s.residual = 1;
              s.cres = Zr;
            }
          }
        }
        s.Zr = Zr;
        s.j = j;
      }
      __syncthreads();
    }
    const int acc = s.accepted;
    if (acc >= 0) {
      if (tid == 0) {
        ot[level] = s.nd_tok[acc];
        on[level] = acc;
      }
      node = acc;
      ++level;
      __syncthreads();
      continue;
    }

    // 4. the bonus from the final residual, in id order
    float Zr = s.Zr;
    const bool empty = s.empty || !(Zr > 0.0f);
    const bool residual = s.residual && !empty;
    const float cres = s.cres, dmax = s.dmax, qscale = s.qscale;
    const int nz = empty ? 0 : s.nzero;
    if (empty) Zr = 1.0f;
    if (tid == 0) {
      s.bonus = -1;
      s.bonus_last = -1;
      s.bonus_target = static_cast<double>(L.u_bonus[b]) * static_cast<double>(Zr);
      if (empty && (s.empty || s.residual || s.nzero > 0)) set_status(L.status, SPEC_TREE_S_RESIDUAL_EMPTY);
    }
    __syncthreads();
    const double target = s.bonus_target;
    const float tie = VD_MARGIN * Zr;
    double carry = 0.0;
    const int rounds = (nvec + VD_THREADS - 1) / VD_THREADS + 1;  // the last round: the scalar tail
    for (int r = 0; r < rounds; ++r) {
      float w[E::VEC];
      int id0 = 0, nel = 0;
      if (r + 1 < rounds) {
        const int vi = r * VD_THREADS + tid;
        id0 = vi * E::VEC;
        if (vi < nvec) {
          const uint4 tv = ldg_stream(trow + static_cast<int64_t>(vi) * 16);
          uint4 dv = make_uint4(0, 0, 0, 0);
          if (residual) dv = ldg_stream(drow + static_cast<int64_t>(vi) * 16);
          // which of the vector's tokens are zeroed or deterministic: the short
          // lists are read once per vector, not once per token
          unsigned zmask = 0u, dmask = 0u;
          for (int k = 0; k < nz; ++k) {
            const unsigned o = static_cast<unsigned>(s.zero[k] - id0);
            if (o < static_cast<unsigned>(E::VEC)) zmask |= 1u << o;
          }
          if (residual)
            for (int k = 0; k < m; ++k) {
              const unsigned o = static_cast<unsigned>(s.det[k] - id0);
              if (o < static_cast<unsigned>(E::VEC)) dmask |= 1u << o;
            }
#pragma unroll
          for (int q = 0; q < E::VEC; ++q) {
            float a = (zmask >> q) & 1u ? 0.0f : vd_ex2((E::get(tv, q) - M) * c) * invZp;
            if (residual && !((dmask >> q) & 1u))
              a = fmaxf(0.0f, a - cres * vd_ex2((E::get(dv, q) - dmax) * c) * qscale);
            w[q] = a;
          }
          nel = E::VEC;
        }
      } else {
        const int id = nvec * E::VEC + tid;
        id0 = id;
        if (id < V) {
          float a = in_list(s.zero, nz, id) ? 0.0f : vd_ex2((E::load(trow, id) - M) * c) * invZp;
          if (residual && !in_list(s.det, m, id))
            a = fmaxf(0.0f, a - cres * vd_ex2((E::load(drow, id) - dmax) * c) * qscale);
          w[0] = a;
          nel = 1;
        }
      }
      // the round's masses in float (a round is a small part of the row), the
      // carry of the rounds before in double: the target relative to it
      float ts = 0.0f;
      int lastp = -1;
#pragma unroll
      for (int q = 0; q < E::VEC; ++q)
        if (q < nel) {
          ts += w[q];
          if (w[q] > 0.0f) lastp = id0 + q;
        }
      if (lastp >= 0) atomicMax(&s.bonus_last, lastp);
      // block exclusive scan of ts
      float incl = ts;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) s.red_s[warp] = incl;
      __syncthreads();
      float before = 0.0f, total = 0.0f;
      for (int k = 0; k < VD_WARPS; ++k) {
        const float y = s.red_s[k];
        if (k < warp) before += y;
        total += y;
      }
      before += incl - ts;
      const float rel = static_cast<float>(target - carry);
      if (ts > 0.0f && before <= rel && rel < before + ts) {
        float run = before;
        int pick = -1;
        for (int q = 0; q < nel && pick < 0; ++q) {
          const float nx = run + w[q];
          if (rel < nx) {
            pick = id0 + q;
            if (L.margins && (rel - run < tie || nx - rel < tie)) atomicAdd(L.margins + 1, 1u);
          }
          run = nx;
        }
        if (pick >= 0) atomicMin(reinterpret_cast<unsigned int*>(&s.bonus), static_cast<unsigned int>(pick));
      }
      carry += static_cast<double>(total);
      __syncthreads();
      if (s.bonus >= 0) break;
    }
    if (tid == 0) {
      int bonus = s.bonus;
      if (bonus < 0) bonus = s.bonus_last;  // rounding left the target past the total
      if (bonus < 0) bonus = 0;
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

}  // namespace

cudaError_t launch_verify_dense(const VerifyLaunch& L, cudaStream_t stream) {
  if (L.B == 0) return cudaSuccess;
  const int smem = static_cast<int>(sizeof(VDShared));
  if (L.dtype == SPEC_TREE_BF16) {
    cudaError_t err = cudaFuncSetAttribute(verify_dense_kernel<__nv_bfloat16>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(verify_dense_kernel<__nv_bfloat16>, dim3(L.B), dim3(VD_THREADS), static_cast<size_t>(smem),
                      stream, L);
  }
  cudaError_t err = cudaFuncSetAttribute(verify_dense_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(verify_dense_kernel<float>, dim3(L.B), dim3(VD_THREADS), static_cast<size_t>(smem), stream, L);
}

}  // namespace st
