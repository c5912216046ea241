// Support selection + dual-identity expansion of draft rows (sm_103a).
//
// RheoSampling notes, Method / Key design 1 (top-128 truncation of the draft
// logits) and Key design 2 (top-m deterministic children, probe sampled from
// the renormalised tempered tail, tail masses).
//
// A persistent CTA owns rows; one producer warp streams every row once
// through a ring of shared-memory stages filled by the TMA engine
// (cp.async.bulk, "full" mbarriers with transaction counts, "empty" mbarriers
// released by the consumer warps), so the consumers never wait on a CTA-wide
// barrier per chunk and the next row is already landing while a row's tail
// work runs.
//
//   pass (HBM; a CTA's first row kept in L2 for its gather when no earlier
//     launch left a cut, other rows streamed with an evict-first hint): each
//     consumer thread reduces its four vectors of every chunk to their
//     maximum with one packed bf16x2 tree and writes it, as a 16-bit order
//     key, to a table in shared memory (thread x chunk); it also keeps its
//     running maximum.
//   bound: thread maxima are distinct elements of the row, so if warp w's
//     j-th largest thread maximum is b_w, with j * (consumer warps) >= |S|,
//     then min_w b_w is a lower bound of the |S|-th largest logit.
//   gather: only the (chunk, thread) pairs whose table entry reaches the
//     bound can hold a candidate -- typically ~250 of 4096 per 128K-token
//     row.  They are listed, the list's vectors are re-read with plain loads
//     spread over the whole CTA (one round of loads in flight), and every
//     element that reaches the bound is appended to a candidate buffer of
//     64-bit (order key, ~token id) composites and counted in a histogram of
//     key offsets above the bound.
//   queue (bf16 rows of up to 16 chunks): the cut of the support is nearly
//     the same from row to row, so a threshold a margin below a recent
//     row's cut predicts which vectors can hold a candidate.  During the
//     pass each warp copies every vector whose maximum reaches it into its
//     own queue in shared memory; after the pass the queued vectors are
//     filtered in shared memory, with no re-read.  The prediction is
//     checked exactly: when at least |S| elements reach the threshold, every
//     element that reaches it was queued (a vector holding one has its
//     maximum above it), so the threshold is a valid bound.  Otherwise (a
//     threshold too high, a full queue, a NaN) the row takes the bound and
//     gather above, from the same pass.
//   select (one warp, overlapped with the next row): the histogram gives the
//     |S|-th largest key and the count above it; the candidates are cut to
//     the exact top-|S| by (logit desc, id asc), ranked by a count, and turned
//     into q, q_T, z, z_T and the probe.
//
// Rows whose candidates overflow the buffer (massive ties at the bound), whose
// bound has no value (NaN), or that are longer than the table are redone by a
// robust path that streams the row from global memory in id order, keeping
// the exact top-|S| of the prefix seen and a strict threshold.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#include "st_common.cuh"
#include "st_keys.cuh"
#include "st_kernels.h"
#include "st_epilogue.cuh"

namespace st {

constexpr int SX_MAX_S = 128;                    // supports of up to 128 tokens (larger: select_wide.cu)
constexpr int SX_CONS = 256;                     // streaming consumer threads (8 warps)
constexpr int SX_CWARPS = SX_CONS / 32;
constexpr int SX_SEL_WARP = SX_CWARPS;           // warp 8: exact selection + epilogue
constexpr int SX_PROD_WARP = SX_CWARPS + 1;      // warp 9: bulk-copy producer
constexpr int SX_THREADS = SX_CONS + 64;
constexpr int SX_VPT = 4;                        // 16-byte vectors per consumer thread per stage
constexpr int SX_CHUNK = SX_CONS * 16 * SX_VPT;  // 16 KB per stage
constexpr int SX_STAGES = 5;
constexpr int SX_FB_THREADS = 128;               // robust path: threads reading per step
constexpr int SX_CAP = 640;                      // candidates of one row (64-bit composites)
constexpr int SX_FB_STEP = SX_FB_THREADS * 8;    // robust path: at most this many appends per step
constexpr int SX_FB_CAP = 1792;                  // robust path: candidate storage
constexpr int SX_FB_HIGH = SX_FB_CAP - SX_FB_STEP;
constexpr int SX_TBL = 32;                       // chunk maxima kept per thread: rows of up to 32 chunks
constexpr int SX_GLIST = 1024;                   // gather list: (chunk, thread) pairs whose maximum reaches the bound
constexpr int SX_QCH = 16;                       // queue path: rows of up to this many chunks
constexpr int SX_QW = 56;                        // queue path: vectors queued per warp and row
constexpr uint32_t SX_QMARGIN = 16;              // queue threshold: this many key steps below a recent cut
constexpr int SX_ANN = 8;                        // rows announced by the producer ahead of the consumers
// what the selector receives with a row's candidates
constexpr int SX_HIST = 1;     // every element >= hbase, with its key histogram khist
constexpr int SX_SORTED = 2;   // exactly the top-|S|, in order

// Storage of the robust path (consumer threads), used only after the
// table of chunk maxima, so the two share it.
struct RobustScratch {
  uint64_t fbuf[SX_FB_CAP];
  uint64_t sel[SX_MAX_S];
  uint64_t tie[32];
  uint32_t hist[256];
};

// The queue path's storage: the table of rows of up to SX_QCH chunks, then
// each warp's queued vectors and their vector indices in the row.
struct QueueView {
  uint16_t tbl_lo[SX_QCH][SX_CONS];
  uint4 vec[SX_CWARPS][SX_QW];
  uint16_t vid[SX_CWARPS][SX_QW];
};

struct SelShared {
  alignas(128) uint8_t ring[SX_STAGES][SX_CHUNK];
  uint64_t cand[2][SX_CAP];  // double-buffered candidates: streamers fill one, the selector drains the other
  union {
    uint16_t tbl[SX_TBL][SX_CONS];  // order key of each consumer thread's maximum in each chunk
    RobustScratch rb;
    QueueView qv;
  };
  uint16_t glist[SX_GLIST];  // chunk << 8 | thread
  alignas(16) uint64_t ssel[SX_MAX_S];  // selector's scratch
  uint64_t stie[32];                      // selector's ties
  uint32_t khist[2][256];  // per candidate buffer: histogram of candidate keys above hbase
  uint64_t full[SX_STAGES];
  uint64_t empty[SX_STAGES];
  uint64_t cfull[2];   // candidates of a row ready for the selector
  uint64_t cempty[2];  // selector done with a candidate buffer
  int64_t cand_row[2];  // output row (support arrays) of the candidates
  int64_t cand_in[2];   // input row (logits, u_probe) of the candidates
  uint32_t shist[256];
  uint32_t warp_bound[SX_CWARPS];
  int count[2];
  int mode[2];         // candidates handed over: SX_HIST or SX_SORTED
  uint32_t hbase[2];   // SX_HIST: the bound the candidates reach (bin 0 of khist)
  int glist_n;
  int sel_count;
  int tie_count;
  int radix_bin;
  int radix_above;
  int radix_cnt;
  uint32_t thr_key;
  int strict;
  int timeout;
  uint32_t last_cut;   // key of the |S|-th largest of the selector's latest row (0: none yet)
  uint32_t thr_row[2]; // queue threshold of the rows of each parity (0: no queue)
  int qbad;            // 1 + the last row whose queue failed (NaN, full queue)
  int64_t ann_row[SX_ANN];   // rows announced by the producer, in this CTA's order (-1: no more)
  uint64_t ann_bar[SX_ANN];  // one arrival per announcement
};

// A candidate buffer and its fill count.
struct CandBuf {
  uint64_t* c;
  int* n;
  int cap;
};

// two CTAs per SM: 228 KB of shared memory per SM, 1 KB of it reserved per CTA
static_assert(sizeof(SelShared) <= 233472 / 2 - 1024, "select_expand needs two CTAs per SM");
static_assert(sizeof(QueueView) <= sizeof(RobustScratch) && sizeof(QueueView) <= 2 * SX_TBL * SX_CONS,
              "the queue shares the table's storage");
static_assert(offsetof(QueueView, vec) % 16 == 0, "queued vectors are 16-byte aligned");

size_t select_expand_smem_bytes() { return sizeof(SelShared); }

// Barrier over the consumer warps only (the producer warp never joins).
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(SX_CONS) : "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Running maximum of pass 1, as an order key (0 when the thread saw nothing).
// bf16: packed bf16x2 max that propagates NaN (a thread that saw NaN reports
// key 0, which only lowers the bound, and the row is flagged).  f32: keys.
template <typename T>
struct RunMax;

template <>
struct RunMax<__nv_bfloat16> {
  __nv_bfloat162 m;
  uint32_t extra;  // key of elements folded in one at a time
  bool any;
  __device__ void init() {
    m = __floats2bfloat162_rn(-INFINITY, -INFINITY);
    extra = 0u;
    any = false;
  }
  __device__ void add(const uint4& v) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&v.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&v.w);
    m = __hmax2_nan(m, __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d)));
    any = true;
  }
  // four vectors at once: a balanced tree of packed maxima
  __device__ void add4(const uint4* v) {
    __nv_bfloat162 x[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __nv_bfloat162* w = reinterpret_cast<const __nv_bfloat162*>(&v[q]);
      x[2 * q] = __hmax2_nan(w[0], w[1]);
      x[2 * q + 1] = __hmax2_nan(w[2], w[3]);
    }
    const __nv_bfloat162 y0 = __hmax2_nan(__hmax2_nan(x[0], x[1]), __hmax2_nan(x[2], x[3]));
    const __nv_bfloat162 y1 = __hmax2_nan(__hmax2_nan(x[4], x[5]), __hmax2_nan(x[6], x[7]));
    m = __hmax2_nan(m, __hmax2_nan(y0, y1));
    any = true;
  }
  __device__ void add_key(uint32_t key) {
    extra = max(extra, key);
    any = true;
  }
  __device__ uint32_t key(bool& nonfinite) const {
    if (!any) return 0u;
    const uint32_t lo = __bfloat16_as_ushort(m.x), hi = __bfloat16_as_ushort(m.y);
    if (((lo & 0x7fffu) > 0x7f80u) || ((hi & 0x7fffu) > 0x7f80u)) {
      nonfinite = true;
      return 0u;
    }
    return max(extra, max(bf16_key(lo), bf16_key(hi)));
  }
};

template <>
struct RunMax<float> {
  uint32_t k;
  bool nf;
  __device__ void init() {
    k = 0u;
    nf = false;
  }
  __device__ void add(const uint4& v) {
#pragma unroll
    for (int j = 0; j < 4; ++j) k = max(k, elem_key<float>(v, j, nf));
  }
  __device__ void add4(const uint4* v) {
#pragma unroll
    for (int q = 0; q < 4; ++q) add(v[q]);
  }
  __device__ void add_key(uint32_t key) { k = max(k, key); }
  __device__ uint32_t key(bool& nonfinite) const {
    if (nf) nonfinite = true;
    return k;
  }
};

// Warp-aggregated append of the elements selected by `mask` (bit j: key
// keys[j], id id0 + j).  All 32 lanes of the warp call it.
template <int VEC>
__device__ __forceinline__ void append_warp(CandBuf cb, uint32_t mask, const uint32_t* keys, uint32_t id0,
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
  if (lane == 31) base = atomicAdd(cb.n, total);
  base = __shfl_sync(FULL, base, 31);
  int pos = base + incl - cnt;
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    if (mask & (1u << j)) {
      if (pos < cb.cap) cb.c[pos] = make_comp(keys[j], id0 + j);
      else overflow = true;
      ++pos;
    }
  }
}

// Pass-2 filter of 16-byte vectors against the bound: `pass` tells whether
// any element reaches it; `emit` appends every element that does (one shared
// atomic per lane).  bf16: packed bf16x2 compares against the bound's value,
// which order exactly like the keys for every non-NaN element (NaN compares
// false and sorts last).
template <typename T>
struct Filter;

template <>
struct Filter<__nv_bfloat16> {
  __nv_bfloat162 b2;
  __device__ void init(uint32_t bound) {
    const __nv_bfloat16 bv = __float2bfloat16_rn(bf16_key_value(bound));
    b2 = __halves2bfloat162(bv, bv);
  }
  // element-wise maximum of four vectors (NaN ignored)
  __device__ static __forceinline__ uint4 merge4(const uint4* v) {
    uint4 r;
    uint32_t* o = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const __nv_bfloat162 x0 = reinterpret_cast<const __nv_bfloat162*>(&v[0])[w];
      const __nv_bfloat162 x1 = reinterpret_cast<const __nv_bfloat162*>(&v[1])[w];
      const __nv_bfloat162 x2 = reinterpret_cast<const __nv_bfloat162*>(&v[2])[w];
      const __nv_bfloat162 x3 = reinterpret_cast<const __nv_bfloat162*>(&v[3])[w];
      const __nv_bfloat162 mx = __hmax2(__hmax2(x0, x1), __hmax2(x2, x3));
      o[w] = *reinterpret_cast<const uint32_t*>(&mx);
    }
    return r;
  }
  __device__ __forceinline__ bool pass(const uint4& v) const {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&v.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&v.w);
    __nv_bfloat162 mx = __hmax2(__hmax2(a, b), __hmax2(c, d));
    mx = __hmax2(mx, __lowhigh2highlow(mx));
    return __hbge2(mx, b2);
  }
  // hist (or null): per key offset above hbase, the last bin collecting the rest
  __device__ __forceinline__ void emit(CandBuf cb, const uint4& v, uint32_t id0, bool& overflow,
                                       uint32_t* hist = nullptr, uint32_t hbase = 0) const {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&v.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&v.w);
    const uint32_t m0 = __hge2_mask(a, b2), m1 = __hge2_mask(b, b2);
    const uint32_t m2 = __hge2_mask(c, b2), m3 = __hge2_mask(d, b2);
    const uint32_t mask = (m0 & 1u) | ((m0 >> 15) & 2u) | ((m1 & 1u) << 2) | ((m1 >> 13) & 8u) |
                          ((m2 & 1u) << 4) | ((m2 >> 11) & 0x20u) | ((m3 & 1u) << 6) | ((m3 >> 9) & 0x80u);
    int pos = atomicAdd(cb.n, __popc(mask));
    bool nf = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (mask & (1u << j)) {
        const uint32_t key = elem_key<__nv_bfloat16>(v, j, nf);
        if (pos < cb.cap) cb.c[pos] = make_comp(key, id0 + j);
        else overflow = true;
        if (hist) atomicAdd(&hist[min(key - hbase, 255u)], 1u);
        ++pos;
      }
    }
  }
};

template <>
struct Filter<float> {
  uint32_t bound;
  __device__ void init(uint32_t b) { bound = b; }
  // element-wise maximum of four vectors in key order
  __device__ static __forceinline__ uint4 merge4(const uint4* v) {
    uint4 r;
    uint32_t* o = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t k = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) k = max(k, f32_key(reinterpret_cast<const uint32_t*>(&v[q])[w]));
      o[w] = f32_from_key(k);
    }
    return r;
  }
  __device__ __forceinline__ bool pass(const uint4& v) const {
    bool nf = false;
    uint32_t k = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) k = max(k, elem_key<float>(v, j, nf));
    return k >= bound;
  }
  __device__ __forceinline__ void emit(CandBuf cb, const uint4& v, uint32_t id0, bool& overflow,
                                       uint32_t* hist = nullptr, uint32_t hbase = 0) const {
    bool nf = false;
    uint32_t keys[4], mask = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      keys[j] = elem_key<float>(v, j, nf);
      if (keys[j] >= bound) mask |= 1u << j;
    }
    int pos = atomicAdd(cb.n, __popc(mask));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (mask & (1u << j)) {
        if (pos < cb.cap) cb.c[pos] = make_comp(keys[j], id0 + j);
        else overflow = true;
        if (hist) atomicAdd(&hist[min(keys[j] - hbase, 255u)], 1u);
        ++pos;
      }
    }
  }
};

// j-th largest (1 <= j <= 32, with multiplicity) of the 32 lane values of a
// warp: repeated warp maxima, each round retiring every lane that holds the
// current maximum, so at most j rounds.  0 when fewer than j values are
// nonzero.
__device__ __forceinline__ uint32_t warp_kth_largest(uint32_t key, int j) {
  uint32_t x = key;
  for (int it = 0; it < 32; ++it) {
    const uint32_t m = __reduce_max_sync(FULL, x);
    const int c = __popc(__ballot_sync(FULL, x == m));
    if (j <= c || m == 0u) return m;
    j -= c;
    if (x == m) x = 0u;
  }
  return 0u;
}

// Exact top-k of cb.c[0..n) (distinct composites) sorted descending into
// cb.c[0..min(n,k)); count = min(n,k); when n >= k the strict threshold
// becomes the key of the k-th.  Streamer threads only (robust path).
template <int KEY_BITS>
__device__ void select_topk(SelShared& s, CandBuf cb, int n, int k) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (n > k) {
    // digits: the key bytes, then bits 23..0 of ~id (bits 31..24 of ~id are
    // all ones for ids below 2^24)
    constexpr int NKD = KEY_BITS / 8;
    uint64_t prefix = 0, pmask = 0;
    int need = k;
    bool tie_mode = false;
    const int n_round = (n + SX_CONS - 1) / SX_CONS * SX_CONS;
#pragma unroll 1
    for (int d = 0; d < NKD + 3; ++d) {
      const int sh = d < NKD ? 32 + KEY_BITS - 8 * (d + 1) : 8 * (NKD + 2 - d);
      s.rb.hist[tid] = 0;
      csync();
      for (int i = tid; i < n_round; i += SX_CONS) {
        bool valid = i < n;
        const uint64_t c = valid ? cb.c[i] : 0ull;
        valid = valid && ((c & pmask) == prefix);
        const uint32_t bin = static_cast<uint32_t>(c >> sh) & 0xffu;
        const uint32_t tag = valid ? bin : (0x100u | lane);
        const unsigned peers = __match_any_sync(FULL, tag);
        if (valid && lane == __ffs(peers) - 1) atomicAdd(&s.rb.hist[bin], static_cast<uint32_t>(__popc(peers)));
      }
      csync();
      if (warp == 0) {
        uint32_t h[8], tot = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          h[j] = s.rb.hist[255 - 8 * lane - j];
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
      csync();
      const int bin = s.radix_bin, above = s.radix_above, cnt = s.radix_cnt;
      need -= above;
      prefix |= static_cast<uint64_t>(bin) << sh;
      pmask |= 0xffull << sh;
      if (cnt == need) break;
      if (d == NKD - 1 && cnt <= 32) {
        // a few candidates share the boundary key: one warp keeps the `need`
        // smallest ids among them instead of three more radix passes
        tie_mode = true;
        break;
      }
    }
    if (tid == 0) {
      s.sel_count = 0;
      s.tie_count = 0;
    }
    csync();
    for (int i = tid; i < n; i += SX_CONS) {
      const uint64_t c = cb.c[i];
      const uint64_t m = c & pmask;
      if (tie_mode ? m > prefix : m >= prefix) {
        const int pos = atomicAdd(&s.sel_count, 1);
        if (pos < SX_MAX_S) s.rb.sel[pos] = c;
      } else if (tie_mode && m == prefix) {
        const int pos = atomicAdd(&s.tie_count, 1);
        if (pos < 32) s.rb.tie[pos] = c;
      }
    }
    csync();
    if (tie_mode && warp == 0) {
      const int nt = min(s.tie_count, 32);
      const uint64_t c = lane < nt ? s.rb.tie[lane] : 0ull;
      int r = 0;
      for (int j = 0; j < nt; ++j) r += s.rb.tie[j] > c;
      if (lane < nt && r < need) {
        const int pos = atomicAdd(&s.sel_count, 1);
        if (pos < SX_MAX_S) s.rb.sel[pos] = c;
      }
    }
    csync();
  } else {
    for (int i = tid; i < n; i += SX_CONS) s.rb.sel[i] = cb.c[i];
    csync();
  }
  const int kk = n < k ? n : k;
  uint64_t c = 0;
  int r = 0;
  if (tid < kk) {
    c = s.rb.sel[tid];
    for (int j = 0; j < kk; ++j) r += (s.rb.sel[j] > c);
  }
  csync();
  if (tid < kk) cb.c[r] = c;
  csync();
  if (tid == 0) {
    *cb.n = kk;
    if (n >= k) {
      s.thr_key = static_cast<uint32_t>(cb.c[kk - 1] >> 32);
      s.strict = 1;
    }
  }
  csync();
}

// Maximum of a consumer thread's four vectors of a chunk (vectors past the
// row given as -inf) as a 16-bit order key for the table, and the full
// order key for the thread's running maximum.  bf16: one packed tree of
// NaN-propagating maxima; a NaN among the elements makes the table entry
// 0xffff (the chunk is examined element by element) and sets nan.  f32: the
// largest element key (NaN excluded, flagged); the table keeps its upper 16
// bits, which order the same way and only ever let more chunks through.
template <typename T>
__device__ __forceinline__ uint32_t chunk_max(const uint4 (&v)[SX_VPT], bool& nan, uint32_t& full);

template <>
__device__ __forceinline__ uint32_t chunk_max<__nv_bfloat16>(const uint4 (&v)[SX_VPT], bool& nan, uint32_t& full) {
  __nv_bfloat162 w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_bfloat162 x0 = reinterpret_cast<const __nv_bfloat162*>(&v[0])[j];
    const __nv_bfloat162 x1 = reinterpret_cast<const __nv_bfloat162*>(&v[1])[j];
    const __nv_bfloat162 x2 = reinterpret_cast<const __nv_bfloat162*>(&v[2])[j];
    const __nv_bfloat162 x3 = reinterpret_cast<const __nv_bfloat162*>(&v[3])[j];
    w[j] = __hmax2_nan(__hmax2_nan(x0, x1), __hmax2_nan(x2, x3));
  }
  __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(w[0], w[1]), __hmax2_nan(w[2], w[3]));
  m = __hmax2_nan(m, __lowhigh2highlow(m));
  const uint32_t bits = __bfloat16_as_ushort(m.x);
  if ((bits & 0x7fffu) > 0x7f80u) {
    nan = true;
    full = 0u;
    return 0xffffu;
  }
  full = bf16_key(bits);
  return full;
}

template <>
__device__ __forceinline__ uint32_t chunk_max<float>(const uint4 (&v)[SX_VPT], bool& nan, uint32_t& full) {
  uint32_t k = 0u;
#pragma unroll
  for (int q = 0; q < SX_VPT; ++q)
#pragma unroll
    for (int j = 0; j < 4; ++j) k = max(k, elem_key<float>(v[q], j, nan));
  full = k;
  return k >> 16;
}

// Queue test: does any element of a 16-byte vector reach the threshold
// (bf16 value, both halves)?  NaN never does.
template <typename T>
__device__ __forceinline__ bool vec_reaches(const uint4& v, __nv_bfloat162 thr2);

template <>
__device__ __forceinline__ bool vec_reaches<__nv_bfloat16>(const uint4& v, __nv_bfloat162 thr2) {
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
  const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&v.z);
  const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&v.w);
  __nv_bfloat162 mx = __hmax2(__hmax2(a, b), __hmax2(c, d));
  mx = __hmax2(mx, __lowhigh2highlow(mx));
  return __hbge2(mx, thr2);
}

template <>
__device__ __forceinline__ bool vec_reaches<float>(const uint4&, __nv_bfloat162) {
  return false;  // f32 rows never take the queue path
}

// Table threshold of a bound: entries at or above it may hold an element >= bound.
template <typename T>
__device__ __forceinline__ uint32_t table_bound(uint32_t bound) {
  return sizeof(T) == 2 ? bound : bound >> 16;
}

struct SelArgs {
  const uint8_t* logits;
  int64_t row_bytes_stride;  // bytes between consecutive rows
  int64_t in_rows;           // rows per tree in the logits / u_probe
  int64_t n_rows;            // rows per tree in the support arrays
  int64_t sup_row0;          // support row of a tree's first processed row
  int64_t rows_used;         // rows per tree to process
  int64_t total_rows;        // B * rows_used
  int V;
  int S;
  int m;
  int draw_probe;
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
  unsigned int* sched;  // [2]: next row to hand out, producers done (NULL: static order)
  unsigned int* hint;   // the cut key of a row of the previous launch (0: none; NULL: not kept)
};

// Robust selection of a row straight from global memory, in id order: keep
// the exact top-|S| of the prefix seen, then only elements strictly above
// its last key (an equal key later in id order loses the tie).
template <typename T>
__device__ void select_row_fallback(SelShared& s, CandBuf cb, const uint8_t* row, int V, int S, bool& nonfinite,
                                    bool& overflow) {
  using E = Elem<T>;
  constexpr int VEC = E::VEC;
  const int tid = threadIdx.x;
  const int nvec = static_cast<int>((static_cast<int64_t>(V) * E::ES) / 16);
  csync();
  if (tid == 0) {
    *cb.n = 0;
    s.thr_key = 0;
    s.strict = 0;
  }
  csync();
  const int steps = (V + SX_FB_THREADS * VEC - 1) / (SX_FB_THREADS * VEC);
  for (int step = 0; step < steps; ++step) {
    const int vi = tid < SX_FB_THREADS ? step * SX_FB_THREADS + tid : 0x7fffffff;
    const uint64_t lo = static_cast<uint64_t>(s.thr_key) + static_cast<uint64_t>(s.strict);
    uint32_t keys[VEC];
    uint32_t mask = 0;
    const uint32_t id0 = static_cast<uint32_t>(vi) * VEC;
    if (vi == 0x7fffffff) {
#pragma unroll
      for (int j = 0; j < VEC; ++j) keys[j] = 0;
    } else if (vi < nvec) {
      const uint4 v = ldg_stream(row + static_cast<int64_t>(vi) * 16);
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        keys[j] = elem_key<T>(v, j, nonfinite);
        if (keys[j] >= lo) mask |= 1u << j;
      }
    } else {
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        keys[j] = 0;
        const int id = static_cast<int>(id0) + j;
        if (id < V) {
          keys[j] = scalar_key<T>(row, id, nonfinite);
          if (keys[j] >= lo) mask |= 1u << j;
        }
      }
    }
    append_warp<VEC>(cb, mask, keys, id0, overflow);
    csync();
    if (*cb.n > SX_FB_HIGH) select_topk<E::KEY_BITS>(s, cb, *cb.n, S);
  }
}

// Bitonic sort, descending, of 32*PER composites held PER per lane
// (element j*32 + lane in val[j]) by one warp.
template <int PER>
__device__ __forceinline__ void warp_bitonic_desc(uint64_t (&val)[PER]) {
  const int lane = threadIdx.x & 31;
  constexpr int N = 32 * PER;
#pragma unroll
  for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
    for (int d = size >> 1; d > 0; d >>= 1) {
      uint64_t nv[PER];
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int e = j * 32 + lane;
        const uint64_t x = val[j];
        const uint64_t y = d >= 32 ? val[j ^ (d >> 5)] : __shfl_xor_sync(FULL, x, d);
        const bool desc = (e & size) == 0;
        const bool lower = (e & d) == 0;
        nv[j] = (desc == lower) ? (x > y ? x : y) : (x < y ? x : y);
      }
#pragma unroll
      for (int j = 0; j < PER; ++j) val[j] = nv[j];
    }
  }
}

// Loads c[0..n) (n <= 32*PER) into PER-per-lane registers padded with 0,
// which sorts below every composite.
template <int PER>
__device__ __forceinline__ void warp_load(const uint64_t* c, int n, uint64_t (&val)[PER]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < PER; ++j) val[j] = j * 32 + lane < n ? c[j * 32 + lane] : 0ull;
}

// Exact radix select of the k largest of c[0..n) into out[0..k) (unordered),
// by one warp with a warp-private histogram (plain shared atomics measured
// faster here than aggregating equal digits with a match first).
template <int KEY_BITS>
__device__ void warp_radix_select(SelShared& s, const uint64_t* c, int n, int k, uint64_t* out) {
  const int lane = threadIdx.x & 31;
  constexpr int NKD = KEY_BITS / 8;
  uint64_t prefix = 0, pmask = 0;
  int need = k;
#pragma unroll 1
  for (int d = 0; d < NKD + 3; ++d) {
    const int sh = d < NKD ? 32 + KEY_BITS - 8 * (d + 1) : 8 * (NKD + 2 - d);
#pragma unroll
    for (int j = 0; j < 8; ++j) s.shist[lane * 8 + j] = 0;
    __syncwarp();
    for (int i0 = 0; i0 < n; i0 += 32) {
      const int i = i0 + lane;
      const uint64_t x = i < n ? c[i] : 0ull;
      const bool valid = i < n && (x & pmask) == prefix;
      const uint32_t bin = static_cast<uint32_t>(x >> sh) & 0xffu;
      if (valid) atomicAdd(&s.shist[bin], 1u);
    }
    __syncwarp();
    uint32_t h[8], tot = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      h[j] = s.shist[255 - 8 * lane - j];
      tot += h[j];
    }
    uint32_t incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += t;
    }
    const uint32_t excl = incl - tot;
    int bin = -1, above = 0, cnt = 0;
    if (excl < static_cast<uint32_t>(need) && static_cast<uint32_t>(need) <= incl) {
      uint32_t acc = excl;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (bin < 0 && acc + h[j] >= static_cast<uint32_t>(need)) {
          bin = 255 - 8 * lane - j;
          above = static_cast<int>(acc);
          cnt = static_cast<int>(h[j]);
        }
        acc += h[j];
      }
    }
    const int src = __ffs(__ballot_sync(FULL, bin >= 0)) - 1;
    bin = __shfl_sync(FULL, bin, src);
    above = __shfl_sync(FULL, above, src);
    cnt = __shfl_sync(FULL, cnt, src);
    need -= above;
    prefix |= static_cast<uint64_t>(bin) << sh;
    pmask |= 0xffull << sh;
    __syncwarp();
    if (cnt == need) break;
  }
  int base = 0;
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int i = i0 + lane;
    const uint64_t x = i < n ? c[i] : 0ull;
    const bool take = i < n && (x & pmask) >= prefix;
    const unsigned bal = __ballot_sync(FULL, take);
    if (take) out[base + __popc(bal & ((1u << lane) - 1u))] = x;
    base += __popc(bal);
  }
  __syncwarp();
}

// Exact top-k (k <= 128) of c[0..n), sorted descending, by one warp: a
// radix select cuts larger sets to k, then a 128-wide register bitonic
// network sorts them.  Returns min(n, k); val[j] holds rank j*32 + lane.
template <int KEY_BITS>
__device__ int warp_select_sort(SelShared& s, const uint64_t* c, int n, int k, uint64_t (&val)[4]) {
  const int kk = n < k ? n : k;
  if (n <= k) {
    warp_load<4>(c, n, val);
  } else {
    warp_radix_select<KEY_BITS>(s, c, n, k, s.ssel);
    warp_load<4>(s.ssel, k, val);
  }
  warp_bitonic_desc<4>(val);
  return kk;
}

// Exact top-k (k <= 128), sorted descending, of candidates that are every
// element of the row with a key >= hbase, given their key histogram h (bin b:
// key hbase + b; the last bin also takes every larger key), by one warp.
// The histogram gives the k-th largest key t and the count above it; keys
// above t are in, and of the keys equal to t the smallest ids fill the rest.
// A counting sort over the histogram's bins then orders the k (descending
// key), and inside a bin a count of larger composites orders them (ascending
// id; the open last bin holds several keys).  Falls back to warp_select_sort
// when t falls in the open last bin or more than 32 keys tie at t.  The
// histogram is used as the bins' cursors (the caller zeroes it afterwards).
template <int KEY_BITS>
__device__ int warp_hist_select_sort(SelShared& s, const uint64_t* c, int n, int k, uint32_t* h,
                                     uint32_t hbase, uint64_t (&val)[4]) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  uint32_t hv[8], tot = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    hv[j] = h[255 - 8 * lane - j];
    tot += hv[j];
  }
  uint32_t incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t excl = incl - tot, kk = static_cast<uint32_t>(k);
  int bin = -1, above = 0, nt = 0;
  if (excl < kk && kk <= incl) {
    uint32_t acc = excl;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (bin < 0 && kk <= acc + hv[j]) {
        bin = 255 - 8 * lane - j;
        above = static_cast<int>(acc);
        nt = static_cast<int>(hv[j]);
      }
      acc += hv[j];
    }
  }
  const int src = __ffs(__ballot_sync(FULL, bin >= 0)) - 1;
  if (src < 0) return warp_select_sort<KEY_BITS>(s, c, n, k, val);
  bin = __shfl_sync(FULL, bin, src);
  above = __shfl_sync(FULL, above, src);
  nt = __shfl_sync(FULL, nt, src);
  const int need = k - above;
  if (bin == 255 || (nt > 32 && nt != need)) return warp_select_sort<KEY_BITS>(s, c, n, k, val);
  const uint32_t t = hbase + static_cast<uint32_t>(bin);
  const bool all_ties = nt == need;
  int base = 0, nties = 0;
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int i = i0 + lane;
    const uint64_t x = i < n ? c[i] : 0ull;
    const uint32_t key = static_cast<uint32_t>(x >> 32);
    const bool valid = i < n;
    const bool take = valid && (key > t || (key == t && all_ties));
    const bool tie = valid && key == t && !all_ties;
    const unsigned tb = __ballot_sync(FULL, take);
    if (take) s.ssel[base + __popc(tb & lt)] = x;
    base += __popc(tb);
    const unsigned eb = __ballot_sync(FULL, tie);
    if (tie) s.stie[nties + __popc(eb & lt)] = x;
    nties += __popc(eb);
  }
  __syncwarp();
  if (!all_ties) {
    // the `need` smallest ids among the keys equal to t (larger composite = smaller id)
    const uint64_t x = lane < nties ? s.stie[lane] : 0ull;
    int r = 0;
    for (int j = 0; j < nties; ++j) r += s.stie[j] > x;
    const bool take = lane < nties && r < need;
    const unsigned tb = __ballot_sync(FULL, take);
    if (take) s.ssel[base + __popc(tb & lt)] = x;
    base += __popc(tb);
    __syncwarp();
  }
  // bin b (>= the cut's bin) starts at the count of selected candidates in
  // higher bins: the cut's bin holds `need` of its ties, higher bins all of theirs
  {
    uint32_t acc = excl;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int bb = 255 - 8 * lane - j;
      if (bb >= bin) h[bb] = acc;
      acc += hv[j];
    }
  }
  __syncwarp();
  // group the k by bin: each takes the next slot of its bin
  uint64_t* grp = reinterpret_cast<uint64_t*>(s.shist);
  uint64_t x[4];
  int xb[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = j * 32 + lane;
    x[j] = 0ull;
    xb[j] = -1;
    if (r < k) {
      x[j] = s.ssel[r];
      xb[j] = static_cast<int>(min(static_cast<uint32_t>(x[j] >> 32) - hbase, 255u));
      grp[atomicAdd(&h[xb[j]], 1u)] = x[j];
    }
  }
  __syncwarp();
  // inside its bin [end of the next higher bin, end of its own), a candidate's
  // place is the count of larger composites there
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (xb[j] < 0) continue;
    const int lo = xb[j] == 255 ? 0 : static_cast<int>(h[xb[j] + 1]);
    const int hi = static_cast<int>(h[xb[j]]);
    int rk = 0;
    for (int i = lo; i < hi; ++i) rk += grp[i] > x[j];
    s.ssel[lo + rk] = x[j];
  }
  __syncwarp();
  warp_load<4>(s.ssel, k, val);
  __syncwarp();
  return k;
}

template <typename T>
__global__ void __launch_bounds__(SX_THREADS, 2) select_expand_kernel(SelArgs a) {
  using E = Elem<T>;
  constexpr int VEC = E::VEC;
  constexpr int CHUNK_ELEMS = SX_CHUNK / E::ES;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SelShared& s = *reinterpret_cast<SelShared*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const int64_t row_bytes = static_cast<int64_t>(a.V) * E::ES;
  const int64_t tma_bytes = row_bytes & ~static_cast<int64_t>(15);
  const int nch = static_cast<int>((tma_bytes + SX_CHUNK - 1) / SX_CHUNK);
  const int tail_begin = static_cast<int>(tma_bytes / 16) * VEC;
  const int last_nvec = nch > 0 ? static_cast<int>((tma_bytes - static_cast<int64_t>(nch - 1) * SX_CHUNK) / 16) : 0;
  // Rows reach a CTA in the order its producer claims them: its first row is
  // blockIdx.x, later ones come from the shared counter a.sched (dynamic
  // balance: a CTA that runs ahead takes more rows), or blockIdx.x +
  // gridDim.x, ... without one; the producer announces each to the
  // consumers.  Rows without a whole chunk have no producer and take the
  // static order.
  const auto static_row = [&](int64_t lr) -> int64_t {
    const int64_t r = static_cast<int64_t>(blockIdx.x) + lr * gridDim.x;
    return r < a.total_rows ? r : -1;
  };
  const bool announced = nch > 0;

  if (tid == 0) {
    for (int i = 0; i < SX_STAGES; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], SX_CWARPS);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.cfull[i], 1);
      mbar_init(&s.cempty[i], 1);
      s.cand_row[i] = -1;
    }
    for (int i = 0; i < SX_ANN; ++i) {
      mbar_init(&s.ann_bar[i], 1);
      s.ann_row[i] = -1;
    }
    fence_mbar_init();
    s.timeout = 0;
    s.last_cut = 0u;
    s.thr_row[0] = s.thr_row[1] = 0u;
    s.qbad = 0;
    s.count[0] = s.count[1] = 0;
  }
  for (int i = tid; i < 2 * 256; i += SX_THREADS) s.khist[i >> 8][i & 255] = 0u;
  grid_dependency_wait();
  grid_dependents_launch();
  if (tid == 0 && a.hint != nullptr) {
    // the first row's queue threshold from the previous launch's cut (the cut
    // barely moves between rows of a workload; a miss costs the exact path)
    const uint32_t h = *a.hint;
    if (h >= 0x80u + SX_QMARGIN) s.thr_row[0] = h - SX_QMARGIN;
  }
  __syncthreads();  // the last CTA-wide barrier: the roles split below

  if (warp == SX_SEL_WARP) {
    // ------------------------------------------------------------ selector ---
    // Rows in order: wait for the streamers' candidates, select the exact
    // top-|S|, sort, expand, write the outputs, hand the buffer back.
    bool timed_out = false;
    for (int64_t lr = 0;; ++lr) {
      const int q = static_cast<int>(lr & 1);
      if (!mbar_wait(&s.cfull[q], static_cast<uint32_t>((lr >> 1) & 1))) timed_out = true;
      const int64_t out_row = s.cand_row[q], in_row = s.cand_in[q];
      if (out_row < 0) break;  // the consumers have no more rows
      const int n = s.count[q];
      uint64_t val[4];
      int n_sup;
      const int mode = s.mode[q];
      if (mode == SX_SORTED) {
        n_sup = n;
        warp_load<4>(s.cand[q], n, val);
      } else if (mode == SX_HIST) {
        n_sup = warp_hist_select_sort<E::KEY_BITS>(s, s.cand[q], min(n, SX_CAP), a.S, s.khist[q], s.hbase[q], val);
      } else {
        n_sup = warp_select_sort<E::KEY_BITS>(s, s.cand[q], min(n, SX_CAP), a.S, val);
      }
      // the row's cut (the key of its |S|-th largest) predicts the next rows' cuts
      if (n_sup == a.S) {
        const int rl = n_sup - 1;
        const uint64_t vc = (rl >> 5) == 0 ? val[0] : (rl >> 5) == 1 ? val[1] : (rl >> 5) == 2 ? val[2] : val[3];
        const uint64_t cut = __shfl_sync(FULL, vc, rl & 31);
        if (lane == 0) *reinterpret_cast<volatile uint32_t*>(&s.last_cut) = static_cast<uint32_t>(cut >> 32);
      }
      expand_epilogue<T>(val, a, out_row, in_row, n_sup);
      // the histogram and the count start the buffer's next row at zero
#pragma unroll
      for (int j = 0; j < 8; ++j) s.khist[q][j * 32 + lane] = 0u;
      if (lane == 0) s.count[q] = 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.cempty[q]);
    }
    if (timed_out && lane == 0) set_status(a.status, SPEC_TREE_S_TIMEOUT);
    // a cut for the next launch's first rows (one writer)
    if (blockIdx.x == 0 && lane == 0 && a.hint != nullptr && s.last_cut != 0u) *a.hint = s.last_cut;
    return;
  }

  if (warp == SX_PROD_WARP) {
    // ------------------------------------------------------------ producer ---
    if (lane == 0 && nch > 0) {
      // L2 hints: with no cut from an earlier launch a CTA's first row takes
      // the bound-and-gather path, which re-reads a few vectors, so it is kept
      // (evict last); every other row mostly takes the queue path and is read
      // once, so it leaves L2 first (kept rows crowd out the other kernels'
      // data: 0.86 -> 0.92 of the measured bandwidth at 64 trees in the
      // bench's step, and 0.93 -> 0.96 once the first rows follow too)
      const uint64_t keep_first_row = s.thr_row[0] != 0u ? l2_evict_first_policy() : l2_evict_last_policy();
      const uint64_t stream_once = l2_evict_first_policy();
      int st = 0;
      uint32_t phase = 0;
      int64_t g = 0;
      bool timed_out = false;
      // a CTA's first row is its own index (the grid never exceeds the rows),
      // so the stream starts without a round trip; the counter hands out the rest
      const auto claim = [&](int64_t lr) -> int64_t {
        if (a.sched == nullptr || lr == 0) return static_row(lr);
        const int64_t r = static_cast<int64_t>(gridDim.x) + atomicAdd(a.sched, 1u);
        return r < a.total_rows ? r : -1;
      };
      // the next row is claimed three chunks before this row's end: late
      // enough that every CTA has its first row by then, early enough that
      // the claim's round trip hides behind the chunks still in the ring
      const int claim_at = nch > 3 ? nch - 3 : 0;
      int64_t next = claim(0);
      for (int64_t lr = 0;; ++lr) {
        const int64_t r = next;
        s.ann_row[lr & (SX_ANN - 1)] = r;
        mbar_arrive(&s.ann_bar[lr & (SX_ANN - 1)]);  // releases the announcement
        if (r < 0) break;
        const int64_t b = r / a.rows_used, e = r - b * a.rows_used;
        const uint8_t* row = a.logits + (b * a.in_rows + e) * a.row_bytes_stride;
        for (int c = 0; c < nch; ++c, ++g) {
          if (c == claim_at) next = claim(lr + 1);
          // stage reuse: wait until every consumer warp released its last use
          if (g >= SX_STAGES && !mbar_wait(&s.empty[st], phase ^ 1u)) timed_out = true;
          const int64_t off = static_cast<int64_t>(c) * SX_CHUNK;
          const uint32_t bytes = static_cast<uint32_t>(min64(SX_CHUNK, tma_bytes - off));
          mbar_expect_tx(&s.full[st], bytes);
          bulk_g2s(s.ring[st], row + off, bytes, &s.full[st], lr == 0 ? keep_first_row : stream_once);
          if (++st == SX_STAGES) {
            st = 0;
            phase ^= 1u;
          }
        }
      }
      if (a.sched != nullptr) {
        // the last producer to stop claiming leaves the counter at zero for
        // the next launch (no claim of this launch can follow)
        __threadfence();
        if (atomicAdd(a.sched + 1, 1u) == gridDim.x - 1) {
          atomicExch(a.sched, 0u);
          atomicExch(a.sched + 1, 0u);
        }
      }
      // before the producer leaves, every copy it issued has landed (a bounded
      // wait on each stage's last phase): the CTA never exits with a bulk copy
      // still writing into its shared memory, even after a consumer gave up
      for (int j = 0; j < SX_STAGES && j < g; ++j) {
        const int64_t last = ((g - 1 - j) / SX_STAGES) * SX_STAGES + j;
        if (!mbar_wait(&s.full[j], static_cast<uint32_t>((last / SX_STAGES) & 1))) timed_out = true;
      }
      if (timed_out) s.timeout = 1;
    }
    return;
  }

  // -------------------------------------------------------------- consumers ---
  bool nonfinite = false, overflow = false, p2over = false;
  int st = 0;
  uint32_t phase = 0;
  const int jth = (a.S + SX_CWARPS - 1) / SX_CWARPS;
  const bool tabled = nch <= SX_TBL;  // longer rows take the robust path
  const bool has_vec = nch > 1 || tid < last_nvec;  // this thread sees at least one whole vector
  const bool queue_rows = sizeof(T) == 2 && nch <= SX_QCH;  // rows that can take the queue path
  const unsigned lt = (1u << lane) - 1u;
  for (int64_t lr = 0;; ++lr) {
    // candidate buffer of this row (the selector may still drain it from two rows ago)
    const int q = static_cast<int>(lr & 1);
    int64_t r;
    if (announced) {
      if (!mbar_wait(&s.ann_bar[lr & (SX_ANN - 1)], static_cast<uint32_t>((lr >> 3) & 1))) s.timeout = 1;
      r = s.ann_row[lr & (SX_ANN - 1)];
    } else {
      r = static_row(lr);
    }
    if (r < 0) {
      // no more rows: tell the selector, once it is done with the buffer
      if (tid == 0) {
        if (lr >= 2 && !mbar_wait(&s.cempty[q], static_cast<uint32_t>(((lr >> 1) - 1) & 1))) s.timeout = 1;
        s.cand_row[q] = -1;
        mbar_arrive(&s.cfull[q]);
      }
      break;
    }
    const int64_t b = r / a.rows_used, e = r - b * a.rows_used;
    const int64_t out_row = b * a.n_rows + a.sup_row0 + e;
    const int64_t in_row = b * a.in_rows + e;
    const uint8_t* row = a.logits + in_row * a.row_bytes_stride;
    const CandBuf cb{s.cand[q], &s.count[q], SX_CAP};
    uint32_t* const kh = s.khist[q];  // zeroed by the selector once it is done with the buffer

    // the queue threshold of this row (a key; 0: no queue), set before a barrier
    const uint32_t thr = queue_rows ? s.thr_row[q] : 0u;
    const bool qmode = thr >= 0x80u;  // smaller keys are NaN patterns
    __nv_bfloat162 thr2;
    {
      const __nv_bfloat16 tv = __float2bfloat16_rn(bf16_key_value(qmode ? thr : 0xffffu));
      thr2 = __halves2bfloat162(tv, tv);
    }
    int qn = 0;  // vectors this warp queued (uniform over the warp)

    // the one pass over the row: each thread's maximum in every chunk goes
    // to the table, and its running maximum is kept; in queue mode every
    // vector whose maximum reaches the threshold is queued by its warp
    uint32_t tkey = 0u;
    bool row_nan = false;
    for (int c = 0; c < nch; ++c) {
      if (!mbar_wait(&s.full[st], phase)) s.timeout = 1;
      const int nvec = c + 1 < nch ? SX_CHUNK / 16 : last_nvec;
      const uint4* src = reinterpret_cast<const uint4*>(s.ring[st]) + tid;
      uint4 v[SX_VPT];
      if (c + 1 < nch) {
#pragma unroll
        for (int k = 0; k < SX_VPT; ++k) v[k] = src[k * SX_CONS];
      } else {
        const uint32_t ninf = sizeof(T) == 2 ? 0xff80ff80u : 0xff800000u;
#pragma unroll
        for (int k = 0; k < SX_VPT; ++k)
          v[k] = tid + k * SX_CONS < nvec ? src[k * SX_CONS] : make_uint4(ninf, ninf, ninf, ninf);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.empty[st]);
      uint32_t full;
      const uint32_t ck = chunk_max<T>(v, row_nan, full);
      tkey = max(tkey, full);
      if (tabled) s.tbl[c][tid] = static_cast<uint16_t>(ck);
      if (qmode) {
#pragma unroll
        for (int k = 0; k < SX_VPT; ++k) {
          const bool hit = vec_reaches<T>(v[k], thr2);
          const unsigned bal = __ballot_sync(FULL, hit);
          if (bal) {
            const int pos = qn + __popc(bal & lt);
            if (hit && pos < SX_QW) {
              s.qv.vec[warp][pos] = v[k];
              s.qv.vid[warp][pos] = static_cast<uint16_t>(c * (SX_CHUNK / 16) + tid + k * SX_CONS);
            }
            qn += __popc(bal);
          }
        }
      }
      if (++st == SX_STAGES) {
        st = 0;
        phase ^= 1u;
      }
    }
    const int tail_id = tail_begin + tid;  // elements past the last whole vector
    uint32_t tail_key = 0u;
    if (tail_id < a.V) tail_key = scalar_key<T>(row, tail_id, row_nan);
    nonfinite = nonfinite || row_nan;
    // a thread's maximum as an order key; 0 (no value) for a thread that saw
    // nothing, or a NaN among bf16 elements (its real maximum is unknown)
    uint32_t tmax = has_vec ? tkey : 0u;
    if (sizeof(T) == 2 && row_nan) tmax = 0u;
    tmax = max(tmax, tail_key);

    bool done = false;  // the row's candidates are complete
    if (qmode) {
      // the buffer's count and histogram were zeroed by the selector when it
      // handed the buffer back two rows ago
      if (lr >= 2 && !mbar_wait(&s.cempty[q], static_cast<uint32_t>(((lr >> 1) - 1) & 1))) s.timeout = 1;
      if (row_nan || qn > SX_QW) s.qbad = static_cast<int>(lr) + 1;
      // filter this warp's queue in shared memory: every element that
      // reaches the threshold becomes a candidate
      Filter<T> flt;
      flt.init(thr);
      const int nq = min(qn, SX_QW);
      for (int i = lane; i < nq; i += 32)
        flt.emit(cb, s.qv.vec[warp][i], static_cast<uint32_t>(s.qv.vid[warp][i]) * VEC, p2over, kh, thr);
      if (tail_id < a.V && tail_key >= thr) {
        const int pos = atomicAdd(cb.n, 1);
        if (pos < cb.cap) cb.c[pos] = make_comp(tail_key, static_cast<uint32_t>(tail_id));
        atomicAdd(&kh[min(tail_key - thr, 255u)], 1u);
      }
      if (tid == 0) {
        // the next row's threshold: a margin below the latest cut (the slot
        // of the other parity, read by the next row after a barrier)
        const uint32_t lc = *reinterpret_cast<volatile uint32_t*>(&s.last_cut);
        s.thr_row[q ^ 1] = lc >= 0x80u + SX_QMARGIN ? lc - SX_QMARGIN : thr;
      }
      csync();
      const int n = *cb.n;
      done = s.qbad != static_cast<int>(lr) + 1 && n >= a.S && n <= SX_CAP;
      if (done) {
        // at least |S| elements reach the threshold, and all of them are
        // here: the selector cuts them with the histogram
        if (tid == 0) {
          s.mode[q] = SX_HIST;
          s.hbase[q] = thr;
        }
      } else {
        // start the row over on the bound-and-gather path
        kh[tid] = 0u;
      }
    }
    if (!done) {
      // the bound: the minimum over warps of each warp's jth-largest thread
      // maximum.  Thread maxima are distinct elements of the row and
      // jth * warps >= |S|, so at least |S| elements reach it.
      const uint32_t wv = warp_kth_largest(tmax, jth);
      if (lane == 0) s.warp_bound[warp] = wv;
      if (tid == 0) {
        if (lr >= 2 && !mbar_wait(&s.cempty[q], static_cast<uint32_t>(((lr >> 1) - 1) & 1))) s.timeout = 1;
        *cb.n = 0;
        s.glist_n = 0;
      }
      csync();
      uint32_t bound = 0xffffffffu;
#pragma unroll
      for (int w = 0; w < SX_CWARPS; ++w) bound = min(bound, s.warp_bound[w]);
      if (tid == 0 && queue_rows) {
        // the next row's threshold: a margin below the latest cut, else this
        // row's bound
        const uint32_t lc = *reinterpret_cast<volatile uint32_t*>(&s.last_cut);
        s.thr_row[q ^ 1] = lc >= 0x80u + SX_QMARGIN ? lc - SX_QMARGIN : bound;
      }
      // a key-0 bound (NaN, or too few elements) has no value to compare against
      bool robust = bound == 0u || !tabled;
      if (!robust) {
        // the gather list: every (chunk, thread) whose maximum reaches the
        // bound (warp-aggregated appends)
        const uint32_t tb = table_bound<T>(bound);
        uint32_t hits = 0u;
        for (int c = 0; c < nch; ++c) hits |= (static_cast<uint32_t>(s.tbl[c][tid]) >= tb ? 1u : 0u) << c;
        const int nh = __popc(hits);
        int incl = nh;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(FULL, incl, o);
          if (lane >= o) incl += y;
        }
        int gbase = 0;
        if (lane == 31) gbase = atomicAdd(&s.glist_n, incl);
        gbase = __shfl_sync(FULL, gbase, 31) + incl - nh;
        while (hits) {
          const int c = __ffs(hits) - 1;
          hits &= hits - 1u;
          if (gbase < SX_GLIST) s.glist[gbase] = static_cast<uint16_t>((c << 8) | tid);
          ++gbase;
        }
        csync();
        const int nlist = s.glist_n;
        robust = nlist > SX_GLIST;  // more than the candidate buffer could hold anyway
      }
      if (!robust) {
        // the gather: the listed vectors are re-read from L2 (each list entry
        // is the four vectors of one thread in one chunk, spread over the CTA
        // so that every load is in flight at once), and every element that
        // reaches the bound is appended to the candidates and counted in the
        // key histogram
        Filter<T> flt;
        flt.init(bound);
        const int ntask = s.glist_n * SX_VPT;
        for (int i0 = 0; i0 < ntask; i0 += SX_CONS * SX_VPT) {
          uint4 v[SX_VPT];
          uint32_t vid[SX_VPT];
          bool ok[SX_VPT];
#pragma unroll
          for (int u = 0; u < SX_VPT; ++u) {
            const int i = i0 + u * SX_CONS + tid;
            ok[u] = false;
            vid[u] = 0u;
            v[u] = make_uint4(0, 0, 0, 0);
            if (i < ntask) {
              const uint32_t ent = s.glist[i / SX_VPT];
              const int c = static_cast<int>(ent >> 8);
              const int vi = static_cast<int>(ent & 0xffu) + (i % SX_VPT) * SX_CONS;
              const int nvec = c + 1 < nch ? SX_CHUNK / 16 : last_nvec;
              ok[u] = vi < nvec;
              vid[u] = static_cast<uint32_t>(c * CHUNK_ELEMS + vi * VEC);
              if (ok[u]) v[u] = ldg_stream(row + static_cast<int64_t>(c) * SX_CHUNK + static_cast<int64_t>(vi) * 16);
            }
          }
#pragma unroll
          for (int u = 0; u < SX_VPT; ++u)
            if (ok[u] && flt.pass(v[u])) flt.emit(cb, v[u], vid[u], p2over, kh, bound);
        }
        if (tail_id < a.V && tail_key >= bound) {
          const int pos = atomicAdd(cb.n, 1);
          if (pos < cb.cap) cb.c[pos] = make_comp(tail_key, static_cast<uint32_t>(tail_id));
          atomicAdd(&kh[min(tail_key - bound, 255u)], 1u);
        }
        csync();
        if (*cb.n <= SX_CAP) {
          // the selector cuts them to the top-|S| with the histogram
          if (tid == 0) {
            s.mode[q] = SX_HIST;
            s.hbase[q] = bound;
          }
        } else {
          robust = true;  // massive ties at the bound
        }
      }
      if (robust) {
        // redo the row in id order from global memory with the robust path's
        // own candidate storage, then hand the selector the exact top-|S|
        const CandBuf fb{s.rb.fbuf, &s.count[q], SX_FB_CAP};
        select_row_fallback<T>(s, fb, row, a.V, a.S, nonfinite, overflow);
        select_topk<E::KEY_BITS>(s, fb, *fb.n, a.S);
        for (int i = tid; i < *fb.n; i += SX_CONS) cb.c[i] = fb.c[i];
        if (tid == 0) s.mode[q] = SX_SORTED;  // select_topk leaves them in order
        csync();
      }
    }
    // hand the candidates to the selector warp and move on to the next row
    if (tid == 0) {
      s.cand_row[q] = out_row;
      s.cand_in[q] = in_row;
      mbar_arrive(&s.cfull[q]);
    }
  }
  if (s.timeout && tid == 0) set_status(a.status, SPEC_TREE_S_TIMEOUT);
  if (nonfinite) set_status(a.status, SPEC_TREE_S_NONFINITE_DRAFT);
  if (overflow) set_status(a.status, SPEC_TREE_S_OVERFLOW);
}

cudaError_t launch_select_expand(int dtype, const SelLaunch& L, cudaStream_t stream) {
  SelArgs a;
  a.logits = static_cast<const uint8_t*>(L.logits);
  a.row_bytes_stride = L.row_stride * (dtype == SPEC_TREE_BF16 ? 2 : 4);
  a.in_rows = L.in_rows;
  a.n_rows = L.n_rows;
  a.sup_row0 = L.sup_row0;
  a.rows_used = L.rows_used;
  a.total_rows = static_cast<int64_t>(L.B) * L.rows_used;
  a.V = L.V;
  a.S = L.S;
  a.m = L.m;
  a.draw_probe = L.draw_probe ? 1 : 0;
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
  // as many CTAs as give every CTA the same number of rows (e.g. 456 rows
  // on 228 CTAs, two each, rather than on 304 with a second wave of 152 rows
  // streamed by half the CTAs, too few bytes in flight to fill the HBM)
  const int64_t max_ctas = static_cast<int64_t>(L.num_sms) * L.ctas_per_sm;
  const int64_t per_cta = (a.total_rows + max_ctas - 1) / max_ctas;
  const int64_t grid = (a.total_rows + per_cta - 1) / per_cta;
  // rows on demand once a CTA has several; with one or two rows a CTA the
  // fixed order spreads the second rows evenly over the SMs
  a.sched = a.total_rows >= 4 * grid ? reinterpret_cast<unsigned int*>(L.sched) : nullptr;
  a.hint = L.sched != nullptr ? reinterpret_cast<unsigned int*>(L.sched) + 2 : nullptr;
  if (dtype == SPEC_TREE_BF16) {
    cudaError_t err = cudaFuncSetAttribute(select_expand_kernel<__nv_bfloat16>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_pdl(select_expand_kernel<__nv_bfloat16>, dim3(static_cast<unsigned>(grid)), dim3(SX_THREADS), smem,
                      stream, a);
  } else {
    cudaError_t err = cudaFuncSetAttribute(select_expand_kernel<float>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_pdl(select_expand_kernel<float>, dim3(static_cast<unsigned>(grid)), dim3(SX_THREADS), smem, stream,
                      a);
  }
}

}  // namespace st
