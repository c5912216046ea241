// Support selection + dual-identity expansion of draft rows (sm_103a).
//
// RheoSampling notes, Method / Key design 1 (top-128 truncation of the draft
// logits) and Key design 2 (top-m deterministic children, probe sampled from
// the renormalised tempered tail, tail masses).
//
// One persistent CTA streams whole rows through a ring of shared-memory stages
// filled by the TMA engine (cp.async.bulk, completion on mbarriers).  While a
// row streams, a rising threshold keeps only elements that can still be in the
// row's top-|S|: every 16-byte vector is first tested with three bf16x2 max
// instructions against the threshold, and only vectors that pass are split
// into elements and appended (warp-aggregated) to a candidate buffer.  When
// the buffer grows past SEL_HIGH, an exact radix select over 64-bit
// (order key, ~token id) composites cuts it back to the exact top-|S| of
// everything seen so far, and the threshold becomes the key of its last
// element (strict from then on: a later element with an equal key has a larger
// id and loses the tie).  At the row end the same select gives the exact
// support, which warp 0 turns into q, q_T, z, z_T and the probe while the next
// row's chunks are already landing.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "st_common.cuh"
#include "st_kernels.h"

namespace st {

constexpr int SEL_THREADS = 512;
constexpr int SEL_WARPS = SEL_THREADS / 32;
constexpr int SEL_CHUNK = SEL_THREADS * 16;  // bytes per stage: one 16-byte vector per thread
constexpr int SEL_STAGES = 6;
constexpr int SEL_HIGH = 1024;               // select when the buffer holds more than this
constexpr int SEL_CAP = SEL_HIGH + SEL_CHUNK / 2;  // + one chunk of bf16 elements

struct SelShared {
  alignas(128) uint8_t ring[SEL_STAGES][SEL_CHUNK];
  uint64_t cand[SEL_CAP];
  uint64_t sel[SPEC_TREE_MAX_SUPPORT];
  uint64_t full[SEL_STAGES];
  uint32_t hist[256];
  uint32_t warp_min[SEL_WARPS];
  int count;
  int sel_count;
  uint32_t thr_key;
  int strict;
  int radix_bin;
  int radix_above;
  int radix_cnt;
  int timeout;
};

size_t select_expand_smem_bytes() { return sizeof(SelShared); }

template <typename T>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int VEC = 8;
  static constexpr int KEY_BITS = 16;
  static constexpr int ES = 2;
};
template <>
struct Elem<float> {
  static constexpr int VEC = 4;
  static constexpr int KEY_BITS = 32;
  static constexpr int ES = 4;
};

// key of element j of a 16-byte vector, and whether it is NaN or +inf
template <typename T>
__device__ __forceinline__ uint32_t elem_key(const uint4& v, int j, bool& nonfinite);

template <>
__device__ __forceinline__ uint32_t elem_key<__nv_bfloat16>(const uint4& v, int j, bool& nonfinite) {
  const uint32_t w = (j < 2) ? v.x : (j < 4) ? v.y : (j < 6) ? v.z : v.w;
  const uint32_t bits = (w >> (16 * (j & 1))) & 0xffffu;
  if ((bits & 0x7fffu) >= 0x7f80u && bits != 0xff80u) nonfinite = true;  // NaN or +inf
  return bf16_key(bits);
}

template <>
__device__ __forceinline__ uint32_t elem_key<float>(const uint4& v, int j, bool& nonfinite) {
  const uint32_t bits = (j == 0) ? v.x : (j == 1) ? v.y : (j == 2) ? v.z : v.w;
  if ((bits & 0x7fffffffu) >= 0x7f800000u && bits != 0xff800000u) nonfinite = true;
  return f32_key(bits);
}

// Upper bound of the keys in a vector; NaN maps to the largest key so that
// a vector holding one always takes the element path (which reports it).
template <typename T>
__device__ __forceinline__ uint32_t vec_max_key(const uint4& v);

template <>
__device__ __forceinline__ uint32_t vec_max_key<__nv_bfloat16>(const uint4& v) {
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
  const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&v.z);
  const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&v.w);
  const __nv_bfloat162 mx = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
  const __nv_bfloat16 h = __hmax_nan(mx.x, mx.y);
  const uint32_t bits = __bfloat16_as_ushort(h);
  if ((bits & 0x7fffu) > 0x7f80u) return 0xffffu;
  return bf16_key(bits);
}

template <>
__device__ __forceinline__ uint32_t vec_max_key<float>(const uint4& v) {
  uint32_t k = 0;
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) k = max(k, f32_is_nan(w[j]) ? 0xffffffffu : f32_key(w[j]));
  return k;
}

template <typename T>
__device__ __forceinline__ float key_value(uint32_t key);
template <>
__device__ __forceinline__ float key_value<__nv_bfloat16>(uint32_t key) { return bf16_key_value(key); }
template <>
__device__ __forceinline__ float key_value<float>(uint32_t key) { return __uint_as_float(f32_from_key(key)); }

__device__ __forceinline__ uint64_t make_comp(uint32_t key, uint32_t id) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~id);
}

// Warp-aggregated append of up to VEC accepted elements per lane.
// `mask` bit j set: element j (key keys[j], id id0 + j) is appended.
template <int VEC>
__device__ __forceinline__ void append_warp(SelShared& s, uint32_t mask, const uint32_t* keys, uint32_t id0,
                                            bool& overflow) {
  const int lane = threadIdx.x & 31;
  if (!__any_sync(FULL, mask != 0)) return;
  const int cnt = __popc(mask);
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += t;
  }
  const int total = __shfl_sync(FULL, incl, 31);
  int base = 0;
  if (lane == 31) base = atomicAdd(&s.count, total);
  base = __shfl_sync(FULL, base, 31);
  int pos = base + incl - cnt;
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    if (mask & (1u << j)) {
      if (pos < SEL_CAP) s.cand[pos] = make_comp(keys[j], id0 + j);
      else overflow = true;
      ++pos;
    }
  }
}

// Exact top-k of s.cand[0..n) (distinct composites), sorted descending into
// s.cand[0..min(n,k)).  Sets count, and the strict threshold when n >= k.
// Called by all threads of the CTA.
template <int KEY_BITS>
__device__ void select_topk(SelShared& s, int n, int k) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (n > k) {
    // digit positions: the key (bits 32..32+KEY_BITS-1), then ~id bits 23..0
    // (bits 31..24 of ~id are all ones for ids below 2^24)
    constexpr int NKD = KEY_BITS / 8;
    int shifts[NKD + 3];
#pragma unroll
    for (int i = 0; i < NKD; ++i) shifts[i] = 32 + KEY_BITS - 8 * (i + 1);
    shifts[NKD] = 16;
    shifts[NKD + 1] = 8;
    shifts[NKD + 2] = 0;
    uint64_t prefix = 0, pmask = 0;
    int need = k;
    const int n_round = (n + SEL_THREADS - 1) / SEL_THREADS * SEL_THREADS;
#pragma unroll 1
    for (int d = 0; d < NKD + 3; ++d) {
      const int sh = shifts[d];
      if (tid < 256) s.hist[tid] = 0;
      __syncthreads();
      for (int i = tid; i < n_round; i += SEL_THREADS) {
        bool valid = i < n;
        const uint64_t c = valid ? s.cand[i] : 0ull;
        valid = valid && ((c & pmask) == prefix);
        const uint32_t bin = static_cast<uint32_t>(c >> sh) & 0xffu;
        const uint32_t tag = valid ? bin : (0x100u | lane);
        const unsigned peers = __match_any_sync(FULL, tag);
        if (valid && lane == __ffs(peers) - 1) atomicAdd(&s.hist[bin], static_cast<uint32_t>(__popc(peers)));
      }
      __syncthreads();
      if (warp == 0) {
        uint32_t h[8], tot = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          h[j] = s.hist[255 - 8 * lane - j];
          tot += h[j];
        }
        uint32_t incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t t = __shfl_up_sync(FULL, incl, o);
          if (lane >= o) incl += t;
        }
        const uint32_t excl = incl - tot;
        if (excl < static_cast<uint32_t>(need) && static_cast<uint32_t>(need) <= incl) {
          uint32_t acc = excl;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (acc + h[j] >= static_cast<uint32_t>(need)) {
              s.radix_bin = 255 - 8 * lane - j;
              s.radix_above = static_cast<int>(acc);
              s.radix_cnt = static_cast<int>(h[j]);
              break;
            }
            acc += h[j];
          }
        }
      }
      __syncthreads();
      const int bin = s.radix_bin, above = s.radix_above, cnt = s.radix_cnt;
      need -= above;
      prefix |= static_cast<uint64_t>(bin) << sh;
      pmask |= 0xffull << sh;
      if (cnt == need) break;
    }
    if (tid == 0) s.sel_count = 0;
    __syncthreads();
    for (int i = tid; i < n; i += SEL_THREADS) {
      const uint64_t c = s.cand[i];
      if ((c & pmask) >= prefix) {
        const int pos = atomicAdd(&s.sel_count, 1);
        if (pos < SPEC_TREE_MAX_SUPPORT) s.sel[pos] = c;
      }
    }
    __syncthreads();
  } else {
    for (int i = tid; i < n; i += SEL_THREADS) s.sel[i] = s.cand[i];
    __syncthreads();
  }
  const int kk = n < k ? n : k;
  uint64_t c = 0;
  int r = 0;
  if (tid < kk) {
    c = s.sel[tid];
    for (int j = 0; j < kk; ++j) r += (s.sel[j] > c);
  }
  __syncthreads();
  if (tid < kk) s.cand[r] = c;
  __syncthreads();
  if (tid == 0) {
    s.count = kk;
    if (n >= k) {
      s.thr_key = static_cast<uint32_t>(s.cand[kk - 1] >> 32);
      s.strict = 1;
    }
  }
  __syncthreads();
}

struct SelArgs {
  const uint8_t* logits;
  int64_t row_bytes_stride;  // bytes between consecutive rows
  int64_t n_rows;            // rows per tree in the logits / support arrays
  int64_t rows_used;         // rows per tree to process
  int64_t total_rows;        // B * rows_used
  int V;
  int S;
  int m;
  float temperature;
  const float* u_probe;
  int32_t* sup_id;
  float* sup_q;
  float* sup_qT;
  float* sup_z;
  float* sup_zT;
  int32_t* probe_pos;
  int sup_stride;
  uint32_t* status;
};

// Softmaxes, tail masses and the probe of one row from its sorted support
// (warp 0).  RheoSampling Key design 2; the probe is the first tail rank k
// with u * z_T < sum_{j=m..k} q_T(j), computed on unnormalised weights.
template <typename T>
__device__ void expand_epilogue(const SelShared& s, const SelArgs& a, int64_t out_row, int n_sup) {
  const int lane = threadIdx.x & 31;
  float l[4];
  uint32_t id[4];
  bool valid[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = 4 * lane + j;
    valid[j] = r < n_sup;
    const uint64_t c = valid[j] ? s.cand[r] : 0ull;
    l[j] = key_value<T>(static_cast<uint32_t>(c >> 32));
    id[j] = ~static_cast<uint32_t>(c);
  }
  const float lmax = __shfl_sync(FULL, l[0], 0);
  if (lane == 0 && !(lmax < INFINITY)) set_status(a.status, SPEC_TREE_S_NONFINITE_DRAFT);
  // weights relative to the row maximum; float32 sums (<= 128 terms, pairwise
  // across lanes) keep the relative error near 1e-7
  float e[4], eT[4];
  float se = 0.0f, seT = 0.0f, te = 0.0f, teT = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = 4 * lane + j;
    const float d = l[j] - lmax;
    e[j] = valid[j] ? expf(d) : 0.0f;
    eT[j] = valid[j] ? expf(d / a.temperature) : 0.0f;
    se += e[j];
    seT += eT[j];
    if (r >= a.m) {
      te += e[j];
      teT += eT[j];
    }
  }
  se = warp_sum(se);
  seT = warp_sum(seT);
  te = warp_sum(te);
  teT = warp_sum(teT);
  int32_t* sid = a.sup_id + out_row * a.sup_stride;
  float* sq = a.sup_q + out_row * a.sup_stride;
  float* sqT = a.sup_qT + out_row * a.sup_stride;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = 4 * lane + j;
    if (valid[j]) {
      sid[r] = static_cast<int32_t>(id[j]);
      sq[r] = e[j] / se;
      sqT[r] = eT[j] / seT;
    }
  }
  int probe = -1;
  if (a.m < n_sup && teT > 0.0f) {
    const float target = a.u_probe[out_row] * teT;
    float cum[4], acc = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (4 * lane + j >= a.m) acc += eT[j];
      cum[j] = acc;
    }
    float incl = acc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += t;
    }
    const float excl = incl - acc;
    int mine = -1, last_pos = -1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = 4 * lane + j;
      if (r >= a.m && valid[j]) {
        if (mine < 0 && target < excl + cum[j]) mine = r;
        if (eT[j] > 0.0f) last_pos = r;
      }
    }
    const unsigned hit = __ballot_sync(FULL, mine >= 0);
    if (hit) {
      probe = __shfl_sync(FULL, mine, __ffs(hit) - 1);
    } else {
      const unsigned pos = __ballot_sync(FULL, last_pos >= 0);
      probe = __shfl_sync(FULL, last_pos, 31 - __clz(pos));
    }
  }
  if (lane == 0) {
    a.sup_z[out_row] = te / se;
    a.sup_zT[out_row] = teT / seT;
    a.probe_pos[out_row] = probe;
  }
}

template <typename T>
__global__ void __launch_bounds__(SEL_THREADS, 2) select_expand_kernel(SelArgs a) {
  using E = Elem<T>;
  constexpr int VEC = E::VEC;
  constexpr int CHUNK_ELEMS = SEL_CHUNK / E::ES;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SelShared& s = *reinterpret_cast<SelShared*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const int64_t row_bytes = static_cast<int64_t>(a.V) * E::ES;
  const int64_t tma_bytes = row_bytes & ~static_cast<int64_t>(15);
  const int nch = static_cast<int>((tma_bytes + SEL_CHUNK - 1) / SEL_CHUNK);
  const int tail_begin = static_cast<int>(tma_bytes / E::ES);
  const int64_t my_rows =
      a.total_rows > blockIdx.x ? (a.total_rows - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int64_t my_chunks = my_rows * nch;

  auto row_ptr = [&](int64_t lr) -> const uint8_t* {
    const int64_t gr = blockIdx.x + lr * gridDim.x;
    const int64_t b = gr / a.rows_used, e = gr % a.rows_used;
    return a.logits + (b * a.n_rows + e) * a.row_bytes_stride;
  };
  const uint64_t policy = l2_evict_first_policy();
  auto issue = [&](int64_t g) {
    const int64_t lr = g / nch;
    const int c = static_cast<int>(g % nch);
    const int64_t off = static_cast<int64_t>(c) * SEL_CHUNK;
    const uint32_t bytes = static_cast<uint32_t>(min64(SEL_CHUNK, tma_bytes - off));
    const int st = static_cast<int>(g % SEL_STAGES);
    mbar_expect_tx(&s.full[st], bytes);
    bulk_g2s(s.ring[st], row_ptr(lr) + off, bytes, &s.full[st], policy);
  };

  if (tid == 0) {
    for (int i = 0; i < SEL_STAGES; ++i) mbar_init(&s.full[i], 1);
    fence_mbar_init();
    s.timeout = 0;
    for (int64_t g = 0; g < my_chunks && g < SEL_STAGES; ++g) issue(g);
  }
  __syncthreads();

  bool nonfinite = false, overflow = false;
  int64_t g = 0;
  for (int64_t lr = 0; lr < my_rows; ++lr) {
    const int64_t gr = blockIdx.x + lr * gridDim.x;
    const int64_t out_row = (gr / a.rows_used) * a.n_rows + gr % a.rows_used;
    if (tid == 0) {
      s.count = 0;
      s.thr_key = 0;
      s.strict = 0;
    }
    __syncthreads();
    for (int c = 0; c < nch; ++c, ++g) {
      const int st = static_cast<int>(g % SEL_STAGES);
      if (!mbar_wait(&s.full[st], static_cast<uint32_t>((g / SEL_STAGES) & 1))) s.timeout = 1;
      const int64_t off = static_cast<int64_t>(c) * SEL_CHUNK;
      const int nvec = static_cast<int>(min64(SEL_CHUNK, tma_bytes - off) / 16);
      const bool have = tid < nvec;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (have) v = *reinterpret_cast<const uint4*>(s.ring[st] + tid * 16);
      const uint32_t id0 = static_cast<uint32_t>(c) * CHUNK_ELEMS + tid * VEC;
      uint64_t lo;
      if (c == 0) {
        // Warm start: 128 groups of 4 lanes; the smallest group maximum is a
        // lower bound of the 128th largest key of the row (each group
        // contributes a distinct element at least that large).
        uint32_t gk = 0u;  // NaN keys are 0 here, so they only lower the bound
        if (have) {
          bool nf = false;
#pragma unroll
          for (int j = 0; j < VEC; ++j) gk = max(gk, elem_key<T>(v, j, nf));
        }
        gk = max(gk, __shfl_xor_sync(FULL, gk, 1));
        gk = max(gk, __shfl_xor_sync(FULL, gk, 2));
        uint32_t wm = gk;
        wm = min(wm, __shfl_xor_sync(FULL, wm, 4));
        wm = min(wm, __shfl_xor_sync(FULL, wm, 8));
        wm = min(wm, __shfl_xor_sync(FULL, wm, 16));
        if (lane == 0) s.warp_min[warp] = wm;
        __syncthreads();
        uint32_t t0 = 0xffffffffu;
#pragma unroll
        for (int w = 0; w < SEL_WARPS; ++w) t0 = min(t0, s.warp_min[w]);
        lo = t0;
        if (tid == 0) s.thr_key = t0;  // still inclusive
      } else {
        lo = static_cast<uint64_t>(s.thr_key) + static_cast<uint64_t>(s.strict);
      }
      uint32_t mask = 0;
      uint32_t keys[VEC];
      if (have && vec_max_key<T>(v) >= lo) {
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
          keys[j] = elem_key<T>(v, j, nonfinite);
          if (keys[j] >= lo) mask |= 1u << j;
        }
      }
      append_warp<VEC>(s, mask, keys, id0, overflow);
      __syncthreads();
      if (tid == 0 && g + SEL_STAGES < my_chunks) {
        fence_proxy_async_smem();
        issue(g + SEL_STAGES);
      }
      if (s.timeout) break;
      if (s.count > SEL_HIGH) select_topk<E::KEY_BITS>(s, s.count, a.S);
    }
    if (s.timeout) break;
    // elements past the last whole 16-byte vector (V not a multiple of VEC)
    if (warp == 0) {
      const int t = tail_begin + lane;
      uint32_t keys[1] = {0u};
      uint32_t mask = 0;
      if (t < a.V) {
        const uint8_t* p = row_ptr(lr) + static_cast<int64_t>(t) * E::ES;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (E::ES == 2) v.x = *reinterpret_cast<const uint16_t*>(p);
        else v.x = *reinterpret_cast<const uint32_t*>(p);
        keys[0] = elem_key<T>(v, 0, nonfinite);
        const uint64_t lo = nch == 0 ? 0ull : static_cast<uint64_t>(s.thr_key) + static_cast<uint64_t>(s.strict);
        if (keys[0] >= lo) mask = 1u;
      }
      append_warp<1>(s, mask, keys, static_cast<uint32_t>(t), overflow);
    }
    __syncthreads();
    const int n = s.count;
    select_topk<E::KEY_BITS>(s, n, a.S);
    if (warp == 0) expand_epilogue<T>(s, a, out_row, n < a.S ? n : a.S);
  }
  if (s.timeout && tid == 0) set_status(a.status, SPEC_TREE_S_TIMEOUT);
  if (nonfinite) set_status(a.status, SPEC_TREE_S_NONFINITE_DRAFT);
  if (overflow) set_status(a.status, SPEC_TREE_S_OVERFLOW);
}

cudaError_t launch_select_expand(int dtype, const SelLaunch& L, cudaStream_t stream) {
  SelArgs a;
  a.logits = static_cast<const uint8_t*>(L.logits);
  a.row_bytes_stride = L.row_stride * (dtype == SPEC_TREE_BF16 ? 2 : 4);
  a.n_rows = L.n_rows;
  a.rows_used = L.rows_used;
  a.total_rows = static_cast<int64_t>(L.B) * L.rows_used;
  a.V = L.V;
  a.S = L.S;
  a.m = L.m;
  a.temperature = L.temperature;
  a.u_probe = L.u_probe;
  a.sup_id = L.sup_id;
  a.sup_q = L.sup_q;
  a.sup_qT = L.sup_qT;
  a.sup_z = L.sup_z;
  a.sup_zT = L.sup_zT;
  a.probe_pos = L.probe_pos;
  a.sup_stride = L.sup_stride;
  a.status = L.status;
  if (a.total_rows == 0) return cudaSuccess;
  const size_t smem = sizeof(SelShared);
  const int64_t grid = min64(a.total_rows, static_cast<int64_t>(L.num_sms) * L.ctas_per_sm);
  if (dtype == SPEC_TREE_BF16) {
    cudaError_t err = cudaFuncSetAttribute(select_expand_kernel<__nv_bfloat16>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    select_expand_kernel<__nv_bfloat16><<<static_cast<unsigned>(grid), SEL_THREADS, smem, stream>>>(a);
  } else {
    cudaError_t err = cudaFuncSetAttribute(select_expand_kernel<float>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    select_expand_kernel<float><<<static_cast<unsigned>(grid), SEL_THREADS, smem, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace st
