// Support selection + dual-identity expansion for supports of 129 to 1024
// tokens (sm_103a): one CTA of SW_THREADS threads per draft row, two per SM.
//
// RheoSampling notes, Method / Key design 1 (the support-size ablation:
// top-128, 256, 512, 1024, and the dense support when it is the whole
// vocabulary) and Key design 2 (softmaxes over the support, tail masses, the
// probe by inverse CDF over the tempered tail in rank order).
//
//   select: an exact radix select on the elements' order keys, one 8-bit
//     digit at a time from the top (two passes over the row for bf16, at most
//     four for f32), each pass counting the elements that match the digits
//     fixed so far into per-warp histograms.  It ends with the |S|-th largest
//     key t and the number of elements equal to t still needed.
//   collect: one more pass, in rounds of SW_THREADS consecutive vectors (token-id
//     order), appends every element above t and, of the elements equal to t,
//     the smallest ids (a block scan ranks them within the round): exactly
//     |S| (key, ~id) composites.
//   sort: a bitonic sort in shared memory, descending, so rank r is thread r.
//   epilogue: q, q_T, z, z_T by block reductions and the probe by a block
//     scan of the tempered tail weights in rank order.
//
// The rows are read from global memory (the first pass from HBM, the others
// mostly from L2); the streaming kernel for supports of up to 128 tokens is
// the fast path.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "st_common.cuh"
#include "st_keys.cuh"
#include "st_kernels.h"
#include "st_epilogue.cuh"

namespace st {

constexpr int SW_THREADS = 512;
constexpr int SW_WARPS = SW_THREADS / 32;
constexpr int SW_MAX_S = SPEC_TREE_MAX_SUPPORT;
constexpr int SW_RPT = (SW_MAX_S + SW_THREADS - 1) / SW_THREADS;  // support ranks a thread owns in the epilogue
constexpr int SW_TBL = 32768;  // table path: rows of up to 32768 vectors (256K bf16 / 128K f32 tokens)
constexpr int SW_CAP = 2048;   // table path: candidates
constexpr int SW_QW = SW_TBL * 2 / 16 / SW_WARPS;  // queue path: vectors queued per warp (the table's storage)

struct WideShared {
  union {
    uint16_t tbl[SW_TBL];  // table path: 16-bit order key of each vector's maximum
    struct {
      uint32_t whist[SW_WARPS][256];                // radix path: per-warp digit histograms
      unsigned long long wmass[SW_WARPS][256];      // dense support: per-warp fixed-point weights
    };
    struct {
      uint64_t grp[SW_CAP];                         // counting sort: candidates grouped by key
      uint32_t cur[SW_CAP];                         //   and each key bin's next free slot
    };
    uint4 qvec[SW_WARPS][SW_QW];                    // queue path: each warp's queued vectors
  };
  uint64_t cand[SW_CAP];            // candidates; at the end the top-|S| in rank order
  union {
    uint32_t list[SW_CAP];            // table path: vectors to gather
    uint16_t qvid[SW_WARPS][SW_QW];   // queue path: the queued vectors' indices in the row
  };
  uint32_t hist[256];
  float red[4][SW_WARPS];         // block reductions
  float scan[SW_RPT][SW_WARPS];   // block scans of the tail weights, one per rank block
  int tie_scan[SW_WARPS];         // block scan of tie counts
  int n_cand;
  int n_list;
  int count;
  int bin;
  int above;
  int cnt;
  int probe;
  int last_pos;
  uint32_t kmin_w[SW_WARPS];  // counting sort: per-warp smallest candidate key
  int sort_ok;
  // dense support
  unsigned long long hmass[256];
  unsigned long long red64[2][SW_WARPS];
  unsigned long long above_mass;
  int nth_id;
  int part_n[8];        // split rows (leader): each part's candidate count, -1 if it declined
  uint32_t part_h[8];   //   and the cut hint it read (the parts must have used one threshold)
};

// Calls f(key, id) for every element of the row that thread tid owns: the
// 16-byte vectors tid, tid + SW_THREADS, ... (loaded eight at a time, so that
// eight loads are in flight) and then the scalar tail element
// nvec * VEC + tid, if any.
template <typename T, typename F>
__device__ __forceinline__ void for_each_elem(const uint8_t* row, int V, int nvec, bool& nonfinite, F f) {
  using E = Elem<T>;
  constexpr int VEC = E::VEC, U = 8;
  const int tid = threadIdx.x;
  for (int v0 = tid; v0 < nvec; v0 += U * SW_THREADS) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int vi = v0 + u * SW_THREADS;
      if (vi < nvec) v[u] = ldg_stream(row + static_cast<int64_t>(vi) * 16);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int vi = v0 + u * SW_THREADS;
      if (vi < nvec)
#pragma unroll
        for (int j = 0; j < VEC; ++j) f(elem_key<T>(v[u], j, nonfinite), static_cast<uint32_t>(vi * VEC + j));
    }
  }
  const int id = nvec * VEC + tid;
  if (id < V) f(scalar_key<T>(row, id, nonfinite), static_cast<uint32_t>(id));
}

// Radix select of the k-th largest key of the row (k >= 1): returns the
// digits fixed (prefix under pmask) and how many elements matching them are
// still needed; *exact is set when every element matching the prefix is in
// (the count of the last bin equalled the need).
template <typename T>
__device__ void radix_select_row(WideShared& s, const uint8_t* row, int V, int nvec, int k, bool& nonfinite,
                                 uint32_t& prefix, uint32_t& pmask, int& need, bool& exact) {
  constexpr int KEY_BITS = Elem<T>::KEY_BITS;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  prefix = 0u;
  pmask = 0u;
  need = k;
  exact = false;
  for (int d = 0; d < KEY_BITS / 8; ++d) {
    const int shift = KEY_BITS - 8 * (d + 1);
#pragma unroll
    for (int i = 0; i < 8; ++i) (&s.whist[0][0])[tid * 8 + i] = 0u;
    __syncthreads();
    uint32_t* wh = s.whist[warp];
    const uint32_t pf = prefix, pm = pmask;
    for_each_elem<T>(row, V, nvec, nonfinite, [&](uint32_t key, uint32_t) {
      if ((key & pm) == pf) atomicAdd(&wh[(key >> shift) & 0xffu], 1u);
    });
    __syncthreads();
    if (tid < 256) {
      uint32_t c = 0;
#pragma unroll 8
      for (int w = 0; w < SW_WARPS; ++w) c += s.whist[w][tid];
      s.hist[tid] = c;
    }
    __syncthreads();
    if (warp == 0) {
      // bins from the top: lane l holds bins 255 - 8l - j
      uint32_t h[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        h[j] = s.hist[255 - 8 * lane - j];
        tot += h[j];
      }
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - tot, nd = static_cast<uint32_t>(need);
      if (excl < nd && nd <= incl) {
        uint32_t acc = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (acc < nd && nd <= acc + h[j]) {
            s.bin = 255 - 8 * lane - j;
            s.above = static_cast<int>(acc);
            s.cnt = static_cast<int>(h[j]);
          }
          acc += h[j];
        }
      }
    }
    __syncthreads();
    need -= s.above;
    prefix |= static_cast<uint32_t>(s.bin) << shift;
    pmask |= 0xffu << shift;
    const bool done = s.cnt == need;
    __syncthreads();  // every thread has read bin, above, cnt
    if (done) {
      exact = true;
      return;
    }
  }
}

// Exclusive block scan of one int per thread; returns the prefix and writes
// the block total to *total.  All threads call it.
__device__ __forceinline__ int block_excl_scan(WideShared& s, int x, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s.tie_scan[warp] = incl;
  __syncthreads();
  int before = 0, tot = 0;
  for (int w = 0; w < SW_WARPS; ++w) {
    const int c = s.tie_scan[w];
    if (w < warp) before += c;
    tot += c;
  }
  __syncthreads();  // tie_scan may be reused
  *total = tot;
  return before + incl - x;
}

// Appends to s.cand every element above the prefix and, unless exact, the
// `need` smallest ids among the elements equal to it (exact: every element
// equal to it).  Rounds of SW_THREADS consecutive vectors keep id order for ties.
template <typename T>
__device__ void collect_row(WideShared& s, const uint8_t* row, int V, int nvec, uint32_t prefix, uint32_t pmask,
                            int need, bool exact, bool& nonfinite) {
  using E = Elem<T>;
  constexpr int VEC = E::VEC;
  const int tid = threadIdx.x;
  if (tid == 0) s.n_cand = 0;
  __syncthreads();
  auto push = [&](uint32_t key, uint32_t id) {
    const int pos = atomicAdd(&s.n_cand, 1);
    if (pos < SW_MAX_S) s.cand[pos] = make_comp(key, id);
  };
  if (exact) {
    for_each_elem<T>(row, V, nvec, nonfinite, [&](uint32_t key, uint32_t id) {
      if ((key & pmask) >= prefix) push(key, id);
    });
    __syncthreads();
    return;
  }
  // ties: key == prefix (every digit fixed); ranked in id order round by round
  int taken = 0;  // ties taken in earlier rounds (block-uniform)
  const int rounds = (nvec + SW_THREADS - 1) / SW_THREADS + 1;  // the last round: the scalar tail
  for (int r = 0; r < rounds; ++r) {
    uint32_t keys[VEC];
    uint32_t id0;
    int nel = 0;
    if (r + 1 < rounds) {
      const int vi = r * SW_THREADS + tid;
      id0 = static_cast<uint32_t>(vi * VEC);
      if (vi < nvec) {
        const uint4 v = ldg_stream(row + static_cast<int64_t>(vi) * 16);
#pragma unroll
        for (int j = 0; j < VEC; ++j) keys[j] = elem_key<T>(v, j, nonfinite);
        nel = VEC;
      }
    } else {
      const int id = nvec * VEC + tid;
      id0 = static_cast<uint32_t>(id);
      if (id < V) {
        keys[0] = scalar_key<T>(row, id, nonfinite);
        nel = 1;
      }
    }
    int ties = 0;
#pragma unroll
    for (int j = 0; j < VEC; ++j)
      if (j < nel) {
        if (keys[j] > prefix) push(keys[j], id0 + j);
        else if (keys[j] == prefix) ++ties;
      }
    int total;
    int rank = block_excl_scan(s, ties, &total) + taken;
#pragma unroll
    for (int j = 0; j < VEC; ++j)
      if (j < nel && keys[j] == prefix) {
        if (rank < need) push(keys[j], id0 + j);
        ++rank;
      }
    taken += total;
    if (taken >= need) {
      // every tie needed is in; the rest of the row is only above-t elements
      for (int r2 = r + 1; r2 + 1 < rounds; ++r2) {
        const int vi = r2 * SW_THREADS + tid;
        if (vi < nvec) {
          const uint4 v = ldg_stream(row + static_cast<int64_t>(vi) * 16);
#pragma unroll
          for (int j = 0; j < VEC; ++j) {
            const uint32_t key = elem_key<T>(v, j, nonfinite);
            if (key > prefix) push(key, static_cast<uint32_t>(vi * VEC + j));
          }
        }
      }
      if (r + 1 < rounds) {
        const int id = nvec * VEC + tid;
        if (id < V) {
          const uint32_t key = scalar_key<T>(row, id, nonfinite);
          if (key > prefix) push(key, static_cast<uint32_t>(id));
        }
      }
      break;
    }
  }
  __syncthreads();
}

// Appends x to buf (when pred) at an index taken from the counter *n, one
// shared atomic per warp (lanes ordered within the warp).  Every lane of the
// warp calls it together.
__device__ __forceinline__ void warp_append(bool pred, uint64_t x, uint64_t* buf, int* n, int cap) {
  const int lane = threadIdx.x & 31;
  const unsigned mask = __ballot_sync(FULL, pred);
  if (mask == 0u) return;
  const int leader = __ffs(mask) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(n, __popc(mask));
  base = __shfl_sync(FULL, base, leader);
  if (pred) {
    const int pos = base + __popc(mask & ((1u << lane) - 1u));
    if (pos < cap) buf[pos] = x;
  }
}

__device__ __forceinline__ void warp_append_u32(bool pred, uint32_t x, uint32_t* buf, int* n, int cap) {
  const int lane = threadIdx.x & 31;
  const unsigned mask = __ballot_sync(FULL, pred);
  if (mask == 0u) return;
  const int leader = __ffs(mask) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(n, __popc(mask));
  base = __shfl_sync(FULL, base, leader);
  if (pred) {
    const int pos = base + __popc(mask & ((1u << lane) - 1u));
    if (pos < cap) buf[pos] = x;
  }
}

// Counting sort of s.cand[0..n) descending.  One bin per key for the keys
// within SW_CAP steps of the smallest candidate key (where nearly all
// candidates sit), and one group, ordered by a rank count, for the few keys
// above them (a row's largest logits, which may lie far away in key space, on
// the other side of zero).  A block scan of the bin counts from the top gives
// each bin's first place after the group; the candidates are grouped by bin,
// and inside a bin (one key) a count of the larger composites orders them by
// id.  Returns false (nothing changed) when the group or a bin holds more than
// 128 candidates; block-uniform.
__device__ bool counting_sort_cand(WideShared& s, int n) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s.sort_ok = 1;
    s.n_list = 0;  // the group's size
  }
  uint32_t kmin = 0xffffffffu;
  for (int i = tid; i < n; i += SW_THREADS) kmin = min(kmin, static_cast<uint32_t>(s.cand[i] >> 32));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) kmin = min(kmin, __shfl_xor_sync(FULL, kmin, o));
  if (lane == 0) s.kmin_w[warp] = kmin;
  for (int b = tid; b < SW_CAP; b += SW_THREADS) s.list[b] = 0u;
  __syncthreads();
  uint32_t kmn = 0xffffffffu;
  for (int w = 0; w < SW_WARPS; ++w) kmn = min(kmn, s.kmin_w[w]);
  // bin b holds key kmn + SW_CAP - 1 - b (bin 0 the largest key in range)
  auto bin_of = [&](uint64_t x) -> int {
    const uint32_t d = static_cast<uint32_t>(x >> 32) - kmn;
    return d < static_cast<uint32_t>(SW_CAP) ? SW_CAP - 1 - static_cast<int>(d) : -1;
  };
  for (int i = tid; i < n; i += SW_THREADS) {
    const int b = bin_of(s.cand[i]);
    if (b >= 0) atomicAdd(&s.list[b], 1u);
    else atomicAdd(&s.n_list, 1);
  }
  __syncthreads();
  const int ng = s.n_list;
  // exclusive scan of the bin counts: thread t owns bins [t*per, (t+1)*per)
  constexpr int per = SW_CAP / SW_THREADS;
  const int b0 = tid * per;
  uint32_t run = 0u, big = 0u;
#pragma unroll
  for (int k = 0; k < per; ++k) {
    run += s.list[b0 + k];
    big = max(big, s.list[b0 + k]);
  }
  int total;
  const int before = block_excl_scan(s, static_cast<int>(run), &total);
  if (big > 128u || ng > 128) s.sort_ok = 0;
  uint32_t acc = static_cast<uint32_t>(ng + before);
#pragma unroll
  for (int k = 0; k < per; ++k) {
    const uint32_t c = s.list[b0 + k];
    s.list[b0 + k] = acc;  // the bin's first place
    s.cur[b0 + k] = acc;
    acc += c;
  }
  if (tid == 0) s.count = 0;  // the group's fill
  __syncthreads();
  if (!s.sort_ok) {
    __syncthreads();
    return false;
  }
  for (int i = tid; i < n; i += SW_THREADS) {
    const uint64_t x = s.cand[i];
    const int b = bin_of(x);
    s.grp[b >= 0 ? static_cast<int>(atomicAdd(&s.cur[b], 1u)) : atomicAdd(&s.count, 1)] = x;
  }
  __syncthreads();
  for (int i = tid; i < n; i += SW_THREADS) {
    const uint64_t x = s.grp[i];
    const int b = bin_of(x);
    const int lo = b >= 0 ? static_cast<int>(s.list[b]) : 0;
    const int hi = b >= 0 ? (b + 1 < SW_CAP ? static_cast<int>(s.list[b + 1]) : n) : ng;
    int rk = 0;
    for (int q = lo; q < hi; ++q) rk += s.grp[q] > x;
    s.cand[lo + rk] = x;
  }
  __syncthreads();
  return true;
}

constexpr int SW_BITONIC_MAX = 2048;  // the largest power of two within SW_CAP

// Sorts s.cand[0..n) descending: the counting sort, else a bitonic sort
// padded with 0 (below every composite) to the next power of two, which needs
// n <= SW_BITONIC_MAX.  Returns false (unsorted) only when neither applies;
// block-uniform.
__device__ bool sort_cand_desc(WideShared& s, int n) {
  if (n > 32 && counting_sort_cand(s, n)) return true;
  if (n > SW_BITONIC_MAX) return false;
  const int tid = threadIdx.x;
  int P = 1;
  while (P < n) P <<= 1;
  for (int i = n + tid; i < P; i += SW_THREADS) s.cand[i] = 0ull;
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int i = tid; i < P / 2; i += SW_THREADS) {
        const int pos = 2 * i - (i & (stride - 1));
        const uint64_t a = s.cand[pos], b = s.cand[pos + stride];
        const bool desc = (pos & size) == 0;
        if ((a < b) == desc) {
          s.cand[pos] = b;
          s.cand[pos + stride] = a;
        }
      }
    }
  }
  __syncthreads();
  return true;
}

// The (r+1)-th largest, with multiplicity, of the 16-bit values x held one
// per thread of the block (0 <= r < blockDim.x): fixes the answer's bits from
// the top, each by one block-wide count of the values that share the bits
// fixed so far and have the next bit set.  All threads call it.
__device__ __forceinline__ uint32_t block_kth_largest_u16(uint32_t x, int r) {
  uint32_t prefix = 0u;
  int need = r + 1;
  for (int bit = 15; bit >= 0; --bit) {
    const uint32_t cand = prefix | (1u << bit);
    const uint32_t hi = 0xffffu & ~((1u << bit) - 1u);
    const int c = __syncthreads_count((x & hi) == cand);
    if (c >= need) prefix = cand;
    else need -= c;
  }
  return prefix;
}

// 16-bit order key of the maximum of one 16-byte vector, for the table:
// bf16: its key (0xffff, so that the vector is examined, when a NaN is among
// the elements); f32: the upper 16 bits of the largest element key, which
// order the same way and only ever let more vectors through.
template <typename T>
__device__ __forceinline__ uint32_t vec_max_key16(const uint4& v, bool& nan);

template <>
__device__ __forceinline__ uint32_t vec_max_key16<__nv_bfloat16>(const uint4& v, bool& nan) {
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
  const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&v.z);
  const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&v.w);
  __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
  m = __hmax2_nan(m, __lowhigh2highlow(m));
  const uint32_t bits = __bfloat16_as_ushort(m.x);
  if ((bits & 0x7fffu) > 0x7f80u) {
    nan = true;
    return 0xffffu;
  }
  return bf16_key(bits);
}

template <>
__device__ __forceinline__ uint32_t vec_max_key16<float>(const uint4& v, bool& nan) {
  uint32_t k = 0u;
#pragma unroll
  for (int j = 0; j < 4; ++j) k = max(k, elem_key<float>(v, j, nan));
  return k >> 16;
}

// Table path: one pass stores every vector's maximum key; the bound is a rank
// of a sample of the table expected to leave about 1.25 |S| entries at
// or above it, accepted once an exact count shows between |S| and SW_CAP
// entries there (each entry is a distinct element, so at least |S| elements
// reach the bound); the listed vectors are re-read and every element that
// reaches the bound becomes a candidate (appended one shared atomic per warp);
// the candidates are sorted (counting sort by key), so the
// first |S| are the top-|S|.  Returns false (nothing decided) when no sample
// rank passes the count, or the candidates are too few (NaN) or too many
// (ties); block-uniform.
template <typename T>
__device__ bool table_select(WideShared& s, const uint8_t* row, int V, int nvec, int S, bool& nonfinite) {
  constexpr int VEC = Elem<T>::VEC, U = 8;
  const int tid = threadIdx.x;
  for (int v0 = tid; v0 < nvec; v0 += U * SW_THREADS) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int vi = v0 + u * SW_THREADS;
      if (vi < nvec) v[u] = ldg_stream(row + static_cast<int64_t>(vi) * 16);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int vi = v0 + u * SW_THREADS;
      if (vi < nvec) s.tbl[vi] = static_cast<uint16_t>(vec_max_key16<T>(v[u], nonfinite));
    }
  }
  __syncthreads();
  const uint32_t sample = s.tbl[static_cast<int64_t>(tid) * nvec / SW_THREADS];
  int r = static_cast<int>(ceilf(1.25f * S * SW_THREADS / nvec)) - 1;
  r = r < 0 ? 0 : (r > SW_THREADS - 1 ? SW_THREADS - 1 : r);
  uint32_t b16 = 0u;
  bool ok = false;
  for (int attempt = 0; attempt < 4 && !ok; ++attempt) {
    b16 = block_kth_largest_u16(sample, r);  // rank r of the sample, in descending order
    int c = 0;
    for (int vi = tid; vi < nvec; vi += SW_THREADS) c += s.tbl[vi] >= b16;
    int total;
    block_excl_scan(s, c, &total);
    if (total >= S && total <= SW_CAP) ok = true;
    else r = total < S ? min(SW_THREADS - 1, 2 * r + 1) : r / 2;
  }
  if (!ok) return false;
  const uint32_t bound = sizeof(T) == 2 ? b16 : (b16 << 16);
  if (tid == 0) {
    s.n_list = 0;
    s.n_cand = 0;
  }
  __syncthreads();
  for (int vb = 0; vb < nvec; vb += SW_THREADS) {  // warp-uniform trip count
    const int vi = vb + tid;
    warp_append_u32(vi < nvec && s.tbl[vi] >= b16, static_cast<uint32_t>(vi), s.list, &s.n_list, SW_CAP);
  }
  __syncthreads();
  const int nl = min(s.n_list, SW_CAP);
  // the listed vectors, two per thread with both loads in flight
  for (int i0 = 0; i0 < nl; i0 += 2 * SW_THREADS) {
    uint4 v[2];
    int vi[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int i = i0 + u * SW_THREADS + tid;
      vi[u] = i < nl ? static_cast<int>(s.list[i]) : -1;
      if (vi[u] >= 0) v[u] = ldg_stream(row + static_cast<int64_t>(vi[u]) * 16);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        const uint32_t key = vi[u] >= 0 ? elem_key<T>(v[u], j, nonfinite) : 0u;
        warp_append(vi[u] >= 0 && key >= bound, make_comp(key, static_cast<uint32_t>(vi[u] * VEC + j)), s.cand,
                    &s.n_cand, SW_CAP);
      }
  }
  const int id = nvec * VEC + tid;  // elements past the last whole vector
  if (id < V) {
    const uint32_t key = scalar_key<T>(row, id, nonfinite);
    if (key >= bound) {
      const int pos = atomicAdd(&s.n_cand, 1);
      if (pos < SW_CAP) s.cand[pos] = make_comp(key, static_cast<uint32_t>(id));
    }
  }
  __syncthreads();
  const int n = s.n_cand;
  if (n < S || n > SW_CAP) return false;
  return sort_cand_desc(s, n);  // false: the radix path takes the row
}

// Queue path (bf16 rows of 2048 to SW_TBL vectors): the cut of the support
// (the key of its |S|-th largest logit) barely moves from row to row of a
// workload, so a threshold a few key steps below the cut of a recent row
// predicts which vectors can hold a candidate.  In the one pass over the row
// each warp copies every vector whose maximum reaches the threshold into its
// own queue in shared memory (a ballot per vector, no atomics); afterwards
// each warp appends the queued elements that reach the threshold as
// candidates, and the candidates are sorted as on the table path.  Exact: a
// vector holding an element that reaches the threshold has its maximum above
// it, so every such element is a candidate, and when at least |S| of them
// exist they hold the top-|S|.  Returns false (nothing decided) when fewer
// than |S| or more than SW_CAP elements reach the threshold, a warp's queue
// overflows or a NaN is seen; the table path then takes the row.
// Block-uniform.
__device__ __forceinline__ uint32_t wide_queue_margin(int S) { return S <= 256 ? 16u : S <= 512 ? 10u : 6u; }

// The queue path's candidates of the vectors [v0, v1) of a row (and, with
// `tail`, of the elements past its last whole vector): every element that
// reaches thr, in s.cand[0..n).  Returns n, or -1 when a warp's queue
// overflows, a NaN is seen or more than SW_CAP elements reach thr.
// Block-uniform.
template <typename T>
__device__ int queue_collect(WideShared& s, const uint8_t* row, int V, int nvec, int v0, int v1, bool tail,
                             uint32_t thr, bool& nonfinite) {
  constexpr int VEC = Elem<T>::VEC, U = 8;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt = (1u << lane) - 1u;
  int nq = 0;  // this warp's queued vectors (warp-uniform)
  bool nan = false;
  for (int vb = v0; vb < v1; vb += U * SW_THREADS) {  // warp-uniform trip count
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int vi = vb + u * SW_THREADS + tid;
      if (vi < v1) v[u] = ldg_stream(row + static_cast<int64_t>(vi) * 16);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int vi = vb + u * SW_THREADS + tid;
      const bool pass = vi < v1 && vec_max_key16<T>(v[u], nan) >= thr;
      const unsigned bal = __ballot_sync(FULL, pass);
      if (bal != 0u) {
        const int slot = nq + __popc(bal & lt);
        if (pass && slot < SW_QW) {
          s.qvec[warp][slot] = v[u];
          s.qvid[warp][slot] = static_cast<uint16_t>(vi);
        }
        nq += __popc(bal);
      }
    }
  }
  if (__syncthreads_or(nan || nq > SW_QW)) return -1;
  // the queued elements that reach the threshold: counted per lane (lane l
  // takes its warp's queued vectors l, l + 32, ...; thread t also the element
  // past the last whole vector, if any), placed by a block scan of the counts
  // and written in order, so no shared counter is contended
  const int id = nvec * VEC + tid;  // elements past the last whole vector
  uint32_t tail_key = 0u;
  if (tail && id < V) tail_key = scalar_key<T>(row, id, nonfinite);
  const bool take_tail = tail && id < V && tail_key >= thr;
  int cnt = take_tail ? 1 : 0;
  for (int i = lane; i < nq; i += 32) {
    const uint4 v = s.qvec[warp][i];
#pragma unroll
    for (int j = 0; j < VEC; ++j) cnt += elem_key<T>(v, j, nonfinite) >= thr;
  }
  int n;
  int pos = block_excl_scan(s, cnt, &n);
  if (n > SW_CAP) return -1;  // block-uniform
  for (int i = lane; i < nq; i += 32) {
    const uint4 v = s.qvec[warp][i];
    const uint32_t id0 = static_cast<uint32_t>(s.qvid[warp][i]) * VEC;
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
      const uint32_t key = elem_key<T>(v, j, nonfinite);
      if (key >= thr) s.cand[pos++] = make_comp(key, id0 + j);
    }
  }
  if (take_tail) s.cand[pos] = make_comp(tail_key, static_cast<uint32_t>(id));
  return n;
}

template <typename T>
__device__ bool queue_select(WideShared& s, const uint8_t* row, int V, int nvec, int S, uint32_t thr,
                             bool& nonfinite) {
  const int n = queue_collect<T>(s, row, V, nvec, 0, nvec, true, thr, nonfinite);
  if (n < S) return false;  // block-uniform (n = -1: declined)
  if (threadIdx.x == 0) s.n_cand = n;
  __syncthreads();
  return sort_cand_desc(s, n);
}

// Softmaxes, tail masses and the probe of a row from its sorted support
// s.cand[0..n): thread t owns support ranks t, t + SW_THREADS, ...
// RheoSampling Key design 2; the probe is the first tail rank k with
// u * z_T < sum_{j=m..k} q_T(j), on unnormalised weights (the last tail rank
// with weight if rounding leaves none).
template <typename T>
__device__ void wide_epilogue(WideShared& s, const SelLaunch& a, int64_t out_row, int64_t in_row, int n) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float lmax = key_value<T>(static_cast<uint32_t>(s.cand[0] >> 32));
  if (tid == 0 && !(lmax < INFINITY)) set_status(a.status, SPEC_TREE_S_NONFINITE_DRAFT);
  uint64_t x[SW_RPT];
  float e[SW_RPT], eT[SW_RPT];
  float v4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int k = 0; k < SW_RPT; ++k) {
    const int r = tid + k * SW_THREADS;
    const bool valid = r < n;
    x[k] = valid ? s.cand[r] : 0ull;
    const float dd = key_value<T>(static_cast<uint32_t>(x[k] >> 32)) - lmax;
    e[k] = valid ? expf(dd) : 0.0f;
    eT[k] = valid ? expf(dd / a.temperature) : 0.0f;
    v4[0] += e[k];
    v4[1] += eT[k];
    if (valid && r >= a.m) {
      v4[2] += e[k];
      v4[3] += eT[k];
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v4[k] = warp_sum(v4[k]);
    if (lane == 0) s.red[k][warp] = v4[k];
  }
  if (tid == 0) {
    s.probe = 0x7fffffff;
    s.last_pos = -1;
  }
  __syncthreads();
  float sum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int w = 0; w < SW_WARPS; ++w)
#pragma unroll
    for (int k = 0; k < 4; ++k) sum[k] += s.red[k][w];
  const float se = sum[0], seT = sum[1], te = sum[2], teT = sum[3];
#pragma unroll
  for (int k = 0; k < SW_RPT; ++k) {
    const int r = tid + k * SW_THREADS;
    if (r < n) {
      a.sup_id[out_row * a.sup_stride + r] = static_cast<int32_t>(~static_cast<uint32_t>(x[k]));
      a.sup_q[out_row * a.sup_stride + r] = e[k] / se;
      a.sup_qT[out_row * a.sup_stride + r] = eT[k] / seT;
    }
  }
  const bool draw = a.draw_probe && a.m < n && teT > 0.0f;  // block-uniform
  if (draw) {
    // inclusive scans of the tail weights in rank order, one per rank block
    float w[SW_RPT], incl[SW_RPT];
#pragma unroll
    for (int k = 0; k < SW_RPT; ++k) {
      const int r = tid + k * SW_THREADS;
      w[k] = (r < n && r >= a.m) ? eT[k] : 0.0f;
      incl[k] = w[k];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(FULL, incl[k], o);
        if (lane >= o) incl[k] += y;
      }
      if (lane == 31) s.scan[k][warp] = incl[k];
    }
    __syncthreads();
    const float target = a.u_probe[in_row] * teT;
    float carry = 0.0f;
#pragma unroll
    for (int k = 0; k < SW_RPT; ++k) {
      const int r = tid + k * SW_THREADS;
      float before = carry, block = 0.0f;
      for (int j = 0; j < SW_WARPS; ++j) {
        const float y = s.scan[k][j];
        if (j < warp) before += y;
        block += y;
      }
      const bool tail = r < n && r >= a.m;
      if (tail && target < before + incl[k]) atomicMin(&s.probe, r);
      if (tail && w[k] > 0.0f) atomicMax(&s.last_pos, r);
      carry += block;
    }
  }
  __syncthreads();
  if (tid == 0) {
    int probe = -1;
    if (draw) probe = s.probe != 0x7fffffff ? s.probe : s.last_pos;
    a.sup_z[out_row] = te / se;
    a.sup_zT[out_row] = teT / seT;
    a.probe_pos[out_row] = probe;
  }
}

// The rest of a row once `done` says whether its exact top-|S| is sorted in
// s.cand: otherwise the table path (rows of 2048 to SW_TBL vectors) and, when
// that declines, the exact radix select; then the row's cut as the next
// rows' hint and the epilogue.
template <typename T>
__device__ void finish_row(WideShared& s, const SelLaunch& a, const uint8_t* row, int nvec, int64_t out_row,
                           int64_t in_row, uint32_t* hint, bool done, bool& nonfinite) {
  const bool tabled = nvec >= 2 * SW_THREADS && nvec <= SW_TBL;
  if (!done && tabled) {
    __syncthreads();  // the queue shares its storage with the table
    done = table_select<T>(s, row, a.V, nvec, a.S, nonfinite);
  }
  if (!done) {
    __syncthreads();  // the table shares its storage with the radix histograms
    uint32_t prefix, pmask;
    int need;
    bool exact;
    radix_select_row<T>(s, row, a.V, nvec, a.S, nonfinite, prefix, pmask, need, exact);
    collect_row<T>(s, row, a.V, nvec, prefix, pmask, need, exact, nonfinite);
    sort_cand_desc(s, min(s.n_cand, a.S));
  }
  const int n = min(s.n_cand, a.S);
  // this row's cut predicts the next rows' (any recent row will do: one
  // plain store, read by CTAs that start later and by the next launch)
  if (threadIdx.x == 0 && hint != nullptr && sizeof(T) == 2 && n == a.S)
    *reinterpret_cast<volatile uint32_t*>(hint) = static_cast<uint32_t>(s.cand[n - 1] >> 32);
  if (a.S <= 128) {
    // the streaming kernel's epilogue, by warp 0: the same supports bit for bit
    if (threadIdx.x < 32) {
      uint64_t val[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = j * 32 + static_cast<int>(threadIdx.x);
        val[j] = r < n ? s.cand[r] : 0ull;
      }
      expand_epilogue<T>(val, a, out_row, in_row, n);
    }
  } else {
    wide_epilogue<T>(s, a, out_row, in_row, n);
  }
  if (nonfinite) set_status(a.status, SPEC_TREE_S_NONFINITE_DRAFT);
}

// A recent row's cut from the row schedule (bf16 rows the queue path can
// take), else 0.
template <typename T>
__device__ __forceinline__ uint32_t read_hint(const uint32_t* hint, int nvec) {
  const bool tabled = nvec >= 2 * SW_THREADS && nvec <= SW_TBL;
  return hint != nullptr && sizeof(T) == 2 && tabled ? *reinterpret_cast<const volatile uint32_t*>(hint) : 0u;
}

template <typename T>
__global__ void __launch_bounds__(SW_THREADS, 2) select_wide_kernel(SelLaunch a, int64_t row_bytes) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  WideShared& s = *reinterpret_cast<WideShared*>(smem_raw);
  const int64_t g = blockIdx.x;
  const int64_t b = g / a.rows_used, e = g % a.rows_used;
  const int64_t out_row = b * a.n_rows + a.sup_row0 + e;
  const int64_t in_row = b * a.in_rows + e;
  grid_dependency_wait();
  grid_dependents_launch();
  const uint8_t* row = static_cast<const uint8_t*>(a.logits) + in_row * row_bytes;
  const int nvec = static_cast<int>((static_cast<int64_t>(a.V) * Elem<T>::ES) / 16);
  bool nonfinite = false;
  // the queue path when a recent row's cut is known, else or when it
  // declines the table path, else the radix select
  uint32_t* hint = a.sched != nullptr ? reinterpret_cast<uint32_t*>(a.sched) + 2 : nullptr;
  const uint32_t h = read_hint<T>(hint, nvec);
  const uint32_t margin = wide_queue_margin(a.S);
  const bool done = h > margin && queue_select<T>(s, row, a.V, nvec, a.S, h - margin, nonfinite);
  finish_row<T>(s, a, row, nvec, out_row, in_row, hint, done, nonfinite);
}

// ------------------------------------------------------------- split rows ---
// Batches with fewer rows than CTA slots: each row is split over a cluster
// of P CTAs.  Every CTA streams its 1/P of the row on the queue path (the
// last one also the elements past the last whole vector) and counts its
// candidates; the counts meet in the leader CTA's shared memory, each CTA
// copies its candidates there behind the others' (distributed shared memory),
// and the leader sorts them and runs the epilogue.  Exact by the queue path's
// argument over the whole row: every element that reaches the threshold is a
// candidate of its part.  When any part declines (no hint, NaN, a full
// queue) or fewer than |S| or more than SW_CAP elements reach the threshold,
// the leader takes the whole row on the table or radix path.
__device__ __forceinline__ uint32_t sw_cluster_addr(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}

template <typename T, int P>
__global__ void __launch_bounds__(SW_THREADS, 2) select_split_kernel(SelLaunch a, int64_t row_bytes) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  WideShared& s = *reinterpret_cast<WideShared*>(smem_raw);
  uint32_t part;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(part));
  const int tid = threadIdx.x;
  const int64_t g = blockIdx.x / P;
  const int64_t b = g / a.rows_used, e = g % a.rows_used;
  const int64_t out_row = b * a.n_rows + a.sup_row0 + e;
  const int64_t in_row = b * a.in_rows + e;
  grid_dependency_wait();
  grid_dependents_launch();
  const uint8_t* row = static_cast<const uint8_t*>(a.logits) + in_row * row_bytes;
  const int nvec = static_cast<int>((static_cast<int64_t>(a.V) * Elem<T>::ES) / 16);
  bool nonfinite = false;
  uint32_t* hint = a.sched != nullptr ? reinterpret_cast<uint32_t*>(a.sched) + 2 : nullptr;
  const uint32_t h = read_hint<T>(hint, nvec);
  const uint32_t margin = wide_queue_margin(a.S);
  int np = -1;  // this part's candidates (-1: declined)
  if (h > margin) {
    const int per = (nvec + P - 1) / P;
    const int v0 = min(static_cast<int>(part) * per, nvec), v1 = min(v0 + per, nvec);
    np = queue_collect<T>(s, row, a.V, nvec, v0, v1, part == P - 1, h - margin, nonfinite);
  }
  if (tid == 0) {
    const uint32_t dn = sw_cluster_addr(&s.part_n[part], 0), dh = sw_cluster_addr(&s.part_h[part], 0);
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(dn), "r"(np) : "memory");
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(dh), "r"(h) : "memory");
  }
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  // a hint another row's leader rewrote between the parts' reads would give
  // the parts different thresholds: then the leader takes the whole row
  int off = 0, total = 0;
  bool ok = true;
#pragma unroll
  for (int q = 0; q < P; ++q) {
    int nq;
    uint32_t hq;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(nq) : "r"(sw_cluster_addr(&s.part_n[q], 0)) : "memory");
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(hq) : "r"(sw_cluster_addr(&s.part_h[q], 0)) : "memory");
    ok = ok && nq >= 0 && hq == h;
    if (q < static_cast<int>(part)) off += nq;
    total += nq;
  }
  ok = ok && total >= a.S && total <= SW_CAP;
  if (ok && part != 0)
    for (int i = tid; i < np; i += SW_THREADS) {
      const uint32_t dst = sw_cluster_addr(&s.cand[off + i], 0);
      asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(dst), "l"(s.cand[i]) : "memory");
    }
  // the candidates are in place, and no CTA writes into another after this
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (part != 0) {
    if (nonfinite) set_status(a.status, SPEC_TREE_S_NONFINITE_DRAFT);
    return;
  }
  bool done = false;
  if (ok) {
    if (tid == 0) s.n_cand = total;
    __syncthreads();
    done = sort_cand_desc(s, total);
  }
  finish_row<T>(s, a, row, nvec, out_row, in_row, hint, done, nonfinite);
}

template <typename T, int P>
cudaError_t launch_split_p(const SelLaunch& L, int64_t row_bytes, cudaStream_t stream) {
  const int smem = static_cast<int>(sizeof(WideShared));
  cudaError_t err = cudaFuncSetAttribute(select_split_kernel<T, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(static_cast<int64_t>(L.B) * L.rows_used * P));
  cfg.blockDim = dim3(SW_THREADS);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = P;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, select_split_kernel<T, P>, L, row_bytes);
}

int select_split_parts(const SelLaunch& L) {
  // the most parts (<= 8) that keep every row's parts in one wave of two
  // CTAs per SM; 1: no split
  const int64_t rows = static_cast<int64_t>(L.B) * L.rows_used;
  const int64_t slots = static_cast<int64_t>(L.num_sms) * 2;
  int p = 8;
  while (p > 1 && rows * p > slots) p /= 2;
  return rows == 0 ? 1 : p;
}

cudaError_t launch_select_split(int dtype, const SelLaunch& L, cudaStream_t stream) {
  // bf16 rows only: the queue path is bf16's
  if (dtype != SPEC_TREE_BF16) return cudaErrorInvalidValue;
  const int P = select_split_parts(L);
  const int64_t rb = L.row_stride * 2;
  if (P >= 8) return launch_split_p<__nv_bfloat16, 8>(L, rb, stream);
  if (P == 4) return launch_split_p<__nv_bfloat16, 4>(L, rb, stream);
  return launch_split_p<__nv_bfloat16, 2>(L, rb, stream);
}

// ------------------------------------------------------------ dense support ---
// |S| = V for a vocabulary of more than SPEC_TREE_MAX_SUPPORT tokens
// (RheoSampling notes, Key design 1: the dense row of the support-size
// ablation; Key design 2 over the whole vocabulary).  One CTA per draft row.
// A row's support arrays hold ranks 0..K-1 (every child but the probe lives
// there: DET ranks 0..m-1, fillers below rank K) and, at entry K, the probe,
// whose rank (probe_pos) may lie anywhere in the tail.
//   ranks 0..K-1: the radix select, collect and sort above with |S| = K;
//   sums: with l_max the rank-0 logit, fixed-point sums (units of 2^-40 of
//     the largest weight) of e = exp(l - l_max) and e_T = exp((l - l_max) / T);
//   probe: the tail's inverse CDF in rank order as a weighted radix select.
//     On the fixed-point scale the target is the DET mass plus u times the
//     tail mass (every DET element precedes every tail element in rank order).
//     One 8-bit digit of the key at a time from the top, per-warp histograms of
//     the weights locate the digit whose cumulative interval holds the target
//     (at the last digit a bin is one key, all of whose elements weigh the
//     same, so counts suffice); the probe is element j, in id order, of that
//     key k*, j = (target - weight above k*) / weight(k*), and its rank is the
//     number of elements above k* plus j.  The weights are integers, so the
//     interval arithmetic is exact: the float32 exponentials are the only
//     rounding.

constexpr float SD_FX_SCALE = 1099511627776.0f;  // 2^40

// Fixed-point weight exp2((l - lmax) * c) in units of 2^-40: at most 2^40, so
// the sum over a row of up to 2^24 elements fits 64 bits.  NaN weighs 0.
__device__ __forceinline__ unsigned long long dense_wfx(float l, float lmax, float c) {
  const float w = exp2f((l - lmax) * c);
  return w > 0.0f ? __float2ull_rn(w * SD_FX_SCALE) : 0ull;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

// Per-thread run of elements that fall in one histogram bin: counted (and
// weighed) once when the run ends, so that the bins most elements share (the
// tail's few exponents) take one shared atomic per run, not per element.
struct BinRun {
  int bin = -1;
  uint32_t cnt = 0u;
  unsigned long long mass = 0ull;
  __device__ __forceinline__ void add(int b, unsigned long long w, uint32_t* wh, unsigned long long* wm) {
    if (b != bin) {
      flush(wh, wm);
      bin = b;
    }
    ++cnt;
    mass += w;
  }
  __device__ __forceinline__ void flush(uint32_t* wh, unsigned long long* wm) {
    if (cnt) atomicAdd(&wh[bin], cnt);
    if (mass) atomicAdd(&wm[bin], mass);
    cnt = 0u;
    mass = 0ull;
  }
};

__device__ __forceinline__ void dense_clear_hist(WideShared& s) {
  for (int i = threadIdx.x; i < SW_WARPS * 256; i += SW_THREADS) {
    (&s.whist[0][0])[i] = 0u;
    (&s.wmass[0][0])[i] = 0ull;
  }
}

// The per-warp histograms summed into s.hist (counts) and s.hmass (weights);
// at the last digit a bin is one key, weighed as its count times its weight.
template <typename T>
__device__ __forceinline__ void dense_reduce_hist(WideShared& s, bool last, uint32_t prefix, int shift, float lmax,
                                                  float c) {
  const int tid = threadIdx.x;
  if (tid < 256) {
    uint32_t cnt = 0u;
    unsigned long long mass = 0ull;
    for (int w = 0; w < SW_WARPS; ++w) {
      cnt += s.whist[w][tid];
      mass += s.wmass[w][tid];
    }
    if (last) mass = cnt ? cnt * dense_wfx(key_value<T>(prefix | (static_cast<uint32_t>(tid) << shift)), lmax, c) : 0ull;
    s.hist[tid] = cnt;
    s.hmass[tid] = mass;
  }
}

// The element at which the fixed-point weight, accumulated in rank order (key
// descending, id ascending), first exceeds `target` (< the row's total): its
// key, the number of elements above that key and their weight.  With
// `level0_ready` the first digit's histograms are in s.hist / s.hmass already.
// All threads call it.
template <typename T>
__device__ void dense_weighted_select(WideShared& s, const uint8_t* row, int V, int nvec, float lmax, float c,
                                      unsigned long long target, bool level0_ready, bool& nonfinite,
                                      uint32_t& key_out, uint32_t& above_cnt, unsigned long long& above_mass) {
  constexpr int KEY_BITS = Elem<T>::KEY_BITS, LEVELS = KEY_BITS / 8;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0u, pmask = 0u, acnt = 0u;
  unsigned long long amass = 0ull;
  for (int d = 0; d < LEVELS; ++d) {
    const int shift = KEY_BITS - 8 * (d + 1);
    const bool last = d == LEVELS - 1;
    if (!(d == 0 && level0_ready)) {
      dense_clear_hist(s);
      __syncthreads();
      uint32_t* wh = s.whist[warp];
      unsigned long long* wm = s.wmass[warp];
      const uint32_t pf = prefix, pm = pmask;
      BinRun run;
      for_each_elem<T>(row, V, nvec, nonfinite, [&](uint32_t key, uint32_t) {
        if ((key & pm) != pf) return;
        run.add(static_cast<int>((key >> shift) & 0xffu), last ? 0ull : dense_wfx(key_value<T>(key), lmax, c), wh, wm);
      });
      run.flush(wh, wm);
      __syncthreads();
      dense_reduce_hist<T>(s, last, prefix, shift, lmax, c);
    }
    if (tid == 0) s.bin = -1;
    __syncthreads();
    if (warp == 0) {
      // bins from the top: lane l holds bins 255 - 8 l - j
      unsigned long long hm[8], tot = 0ull;
      uint32_t hc[8], ctot = 0u;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        hm[j] = s.hmass[255 - 8 * lane - j];
        hc[j] = s.hist[255 - 8 * lane - j];
        tot += hm[j];
        ctot += hc[j];
      }
      unsigned long long incl = tot;
      uint32_t cincl = ctot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(FULL, incl, o);
        const uint32_t cy = __shfl_up_sync(FULL, cincl, o);
        if (lane >= o) {
          incl += y;
          cincl += cy;
        }
      }
      const unsigned long long need = target - amass;
      unsigned long long acc = incl - tot;
      uint32_t cacc = cincl - ctot;
      if (acc <= need && need < incl) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (acc <= need && need < acc + hm[j]) {
            s.bin = 255 - 8 * lane - j;
            s.above_mass = acc;
            s.above = static_cast<int>(cacc);
            s.cnt = static_cast<int>(hc[j]);
          }
          acc += hm[j];
          cacc += hc[j];
        }
      }
    }
    __syncthreads();
    const int bin = s.bin;
    if (bin < 0) break;  // not reached: the target is below the row's total (block-uniform)
    amass += s.above_mass;
    acnt += static_cast<uint32_t>(s.above);
    prefix |= static_cast<uint32_t>(bin) << shift;
    pmask |= 0xffu << shift;
    __syncthreads();  // every thread has read the bin
  }
  key_out = prefix;
  above_cnt = acnt;
  above_mass = amass;
}

// The (r+1)-th largest, with multiplicity, of the KEY_BITS-bit keys x held
// one per thread (0 <= r < blockDim.x), its bits fixed from the top by
// block-wide counts.  All threads call it.
template <int KEY_BITS>
__device__ __forceinline__ uint32_t block_kth_largest_bits(uint32_t x, int r) {
  uint32_t prefix = 0u;
  int need = r + 1;
  for (int bit = KEY_BITS - 1; bit >= 0; --bit) {
    const uint32_t cand = prefix | (1u << bit);
    const uint32_t hi = ~((1u << bit) - 1u);
    const int cnt = __syncthreads_count((x & hi) == cand);
    if (cnt >= need) prefix = cand;
    else need -= cnt;
  }
  return prefix;
}

// Id of element j (0-based, in id order) among the row's elements with order key `key`.
template <typename T>
__device__ int nth_with_key(WideShared& s, const uint8_t* row, int V, int nvec, uint32_t key, int j, bool& nonfinite) {
  constexpr int VEC = Elem<T>::VEC;
  const int tid = threadIdx.x;
  if (tid == 0) s.nth_id = -1;
  __syncthreads();
  int taken = 0;
  const int rounds = (nvec + SW_THREADS - 1) / SW_THREADS + 1;  // the last round: the scalar tail
  for (int r = 0; r < rounds; ++r) {
    uint32_t keys[VEC];
    uint32_t id0;
    int nel = 0;
    if (r + 1 < rounds) {
      const int vi = r * SW_THREADS + tid;
      id0 = static_cast<uint32_t>(vi * VEC);
      if (vi < nvec) {
        const uint4 v = ldg_stream(row + static_cast<int64_t>(vi) * 16);
#pragma unroll
        for (int q = 0; q < VEC; ++q) keys[q] = elem_key<T>(v, q, nonfinite);
        nel = VEC;
      }
    } else {
      const int id = nvec * VEC + tid;
      id0 = static_cast<uint32_t>(id);
      if (id < V) {
        keys[0] = scalar_key<T>(row, id, nonfinite);
        nel = 1;
      }
    }
    int cnt = 0;
#pragma unroll
    for (int q = 0; q < VEC; ++q) cnt += (q < nel && keys[q] == key);
    int total;
    int rank = block_excl_scan(s, cnt, &total) + taken;
    if (rank <= j && j < rank + cnt) {
#pragma unroll
      for (int q = 0; q < VEC; ++q)
        if (q < nel && keys[q] == key) {
          if (rank == j) s.nth_id = static_cast<int>(id0 + q);
          ++rank;
        }
    }
    taken += total;
    if (taken > j) break;
  }
  __syncthreads();
  return s.nth_id;
}

template <typename T>
__global__ void __launch_bounds__(SW_THREADS, 2) select_dense_kernel(SelLaunch a, int64_t row_bytes) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  WideShared& s = *reinterpret_cast<WideShared*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t g = blockIdx.x;
  const int64_t b = g / a.rows_used, e = g % a.rows_used;
  const int64_t out_row = b * a.n_rows + a.sup_row0 + e;
  const int64_t in_row = b * a.in_rows + e;
  grid_dependency_wait();
  grid_dependents_launch();
  const uint8_t* row = static_cast<const uint8_t*>(a.logits) + in_row * row_bytes;
  const int nvec = static_cast<int>((static_cast<int64_t>(a.V) * Elem<T>::ES) / 16);
  bool nonfinite = false;
  const int K = a.S;  // support ranks kept: 0..K-1
  constexpr int KEY_BITS = Elem<T>::KEY_BITS;
  const float c1 = 1.4426950408889634f;
  const float cT = a.temperature == 1.0f ? c1 : c1 / a.temperature;
  const bool same = a.temperature == 1.0f;

  // pass 1 (from HBM): each thread's largest key; the row maximum
  uint32_t tmax = 0u;
  for_each_elem<T>(row, a.V, nvec, nonfinite, [&](uint32_t key, uint32_t) { tmax = max(tmax, key); });
  uint32_t kmax = tmax;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) kmax = max(kmax, __shfl_xor_sync(FULL, kmax, o));
  if (lane == 0) s.hist[warp] = kmax;
  __syncthreads();
  kmax = 0u;
  for (int w = 0; w < SW_WARPS; ++w) kmax = max(kmax, s.hist[w]);
  const float lmax = key_value<T>(kmax);
  // the K-th largest thread maximum: at least K elements reach it (thread maxima are distinct elements)
  const uint32_t bound = block_kth_largest_bits<KEY_BITS>(tmax, K - 1);

  // pass 2: every element at or above the bound as a candidate, the fixed-point
  // sums of e and e_T, and the first digit's weighted histograms for the probe
  if (tid == 0) s.n_cand = 0;
  dense_clear_hist(s);
  __syncthreads();
  unsigned long long se = 0ull, seT = 0ull;
  {
    uint32_t* wh = s.whist[warp];
    unsigned long long* wm = s.wmass[warp];
    BinRun run;
    for_each_elem<T>(row, a.V, nvec, nonfinite, [&](uint32_t key, uint32_t id) {
      const float l = key_value<T>(key);
      const unsigned long long w1 = dense_wfx(l, lmax, c1);
      const unsigned long long wT = same ? w1 : dense_wfx(l, lmax, cT);
      se += w1;
      seT += wT;
      if (key >= bound) {
        const int pos = atomicAdd(&s.n_cand, 1);
        if (pos < SW_CAP) s.cand[pos] = make_comp(key, id);
      }
      run.add(static_cast<int>(key >> (KEY_BITS - 8)), wT, wh, wm);
    });
    run.flush(wh, wm);
  }
  se = warp_sum_u64(se);
  seT = warp_sum_u64(seT);
  if (lane == 0) {
    s.red64[0][warp] = se;
    s.red64[1][warp] = seT;
  }
  __syncthreads();
  se = 0ull;
  seT = 0ull;
  for (int w = 0; w < SW_WARPS; ++w) {
    se += s.red64[0][w];
    seT += s.red64[1][w];
  }
  dense_reduce_hist<T>(s, KEY_BITS == 8, 0u, KEY_BITS - 8, lmax, cT);
  // ranks 0..K-1: the sorted candidates, or (massive ties at the bound) the exact radix path
  const int nc = s.n_cand;
  bool level0_ready = true;
  if (nc >= K && nc <= SW_CAP && sort_cand_desc(s, nc)) {
  } else {
    __syncthreads();  // the radix path reuses the histograms' storage
    uint32_t prefix, pmask;
    int need;
    bool exact;
    radix_select_row<T>(s, row, a.V, nvec, K, nonfinite, prefix, pmask, need, exact);
    collect_row<T>(s, row, a.V, nvec, prefix, pmask, need, exact, nonfinite);
    sort_cand_desc(s, min(s.n_cand, K));
    level0_ready = false;
  }
  const int n = min(level0_ready ? nc : s.n_cand, K);

  // the DET elements (ranks 0..m-1) and their weights
  unsigned long long det1 = 0ull, detT = 0ull;
  for (int r = 0; r < a.m && r < n; ++r) {
    const float l = key_value<T>(static_cast<uint32_t>(s.cand[r] >> 32));
    det1 += dense_wfx(l, lmax, c1);
    detT += dense_wfx(l, lmax, cT);
  }
  const unsigned long long tailT = seT - detT;
  const bool draw = a.draw_probe && a.m < a.V && tailT > 0ull;  // block-uniform
  int probe_rank = -1, probe_id = -1;
  float probe_l = 0.0f;
  if (draw) {
    const float u = a.u_probe[in_row];
    unsigned long long target = detT + static_cast<unsigned long long>(static_cast<double>(u) *
                                                                       static_cast<double>(tailT));
    if (target >= seT) target = seT - 1ull;
    uint32_t kstar, acnt;
    unsigned long long amass;
    dense_weighted_select<T>(s, row, a.V, nvec, lmax, cT, target, level0_ready, nonfinite, kstar, acnt, amass);
    const unsigned long long wk = dense_wfx(key_value<T>(kstar), lmax, cT);
    int j = wk ? static_cast<int>((target - amass) / wk) : 0;
    if (j > s.cnt - 1) j = s.cnt - 1;  // s.cnt: elements of key k*
    if (j < 0) j = 0;
    probe_id = nth_with_key<T>(s, row, a.V, nvec, kstar, j, nonfinite);
    probe_rank = static_cast<int>(acnt) + j;
    probe_l = key_value<T>(kstar);
  }
  const double inv1 = 1.0 / static_cast<double>(se), invT = 1.0 / static_cast<double>(seT);
  const int64_t base = out_row * a.sup_stride;
  for (int r = tid; r < n; r += SW_THREADS) {
    const uint64_t x = s.cand[r];
    const float l = key_value<T>(static_cast<uint32_t>(x >> 32));
    a.sup_id[base + r] = static_cast<int32_t>(~static_cast<uint32_t>(x));
    a.sup_q[base + r] = static_cast<float>(static_cast<double>(dense_wfx(l, lmax, c1)) * inv1);
    a.sup_qT[base + r] = static_cast<float>(static_cast<double>(dense_wfx(l, lmax, cT)) * invT);
  }
  if (tid == 0) {
    a.sup_id[base + K] = probe_id;
    a.sup_q[base + K] = draw ? static_cast<float>(static_cast<double>(dense_wfx(probe_l, lmax, c1)) * inv1) : 0.0f;
    a.sup_qT[base + K] = draw ? static_cast<float>(static_cast<double>(dense_wfx(probe_l, lmax, cT)) * invT) : 0.0f;
    a.sup_z[out_row] = static_cast<float>(static_cast<double>(se - det1) * inv1);
    a.sup_zT[out_row] = static_cast<float>(static_cast<double>(tailT) * invT);
    a.probe_pos[out_row] = draw && probe_id >= 0 ? probe_rank : -1;
    if (!(lmax < INFINITY) || (draw && probe_id < 0)) set_status(a.status, SPEC_TREE_S_NONFINITE_DRAFT);
  }
  if (nonfinite) set_status(a.status, SPEC_TREE_S_NONFINITE_DRAFT);
}

cudaError_t launch_select_dense(int dtype, const SelLaunch& L, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(L.B) * L.rows_used;
  if (rows == 0) return cudaSuccess;
  const int smem = static_cast<int>(sizeof(WideShared));
  if (dtype == SPEC_TREE_BF16) {
    cudaError_t err = cudaFuncSetAttribute(select_dense_kernel<__nv_bfloat16>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(select_dense_kernel<__nv_bfloat16>, dim3(static_cast<unsigned>(rows)), dim3(SW_THREADS),
                      static_cast<size_t>(smem), stream, L, L.row_stride * static_cast<int64_t>(2));
  }
  cudaError_t err = cudaFuncSetAttribute(select_dense_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(select_dense_kernel<float>, dim3(static_cast<unsigned>(rows)), dim3(SW_THREADS),
                    static_cast<size_t>(smem), stream, L, L.row_stride * static_cast<int64_t>(4));
}

cudaError_t launch_select_wide(int dtype, const SelLaunch& L, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(L.B) * L.rows_used;
  if (rows == 0) return cudaSuccess;
  const int smem = static_cast<int>(sizeof(WideShared));
  if (dtype == SPEC_TREE_BF16) {
    cudaError_t err = cudaFuncSetAttribute(select_wide_kernel<__nv_bfloat16>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(select_wide_kernel<__nv_bfloat16>, dim3(static_cast<unsigned>(rows)), dim3(SW_THREADS),
                      static_cast<size_t>(smem), stream, L, L.row_stride * static_cast<int64_t>(2));
  }
  cudaError_t err = cudaFuncSetAttribute(select_wide_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(select_wide_kernel<float>, dim3(static_cast<unsigned>(rows)), dim3(SW_THREADS),
                    static_cast<size_t>(smem), stream, L, L.row_stride * static_cast<int64_t>(4));
}

}  // namespace st
