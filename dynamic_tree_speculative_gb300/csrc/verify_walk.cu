// Layer-by-layer verification of built trees (sm_103a): one thread-block
// cluster of C CTAs per tree.
//
// RheoSampling notes, Method / Key design 3: the probe is tested first with
// min(1, p/q~_T); on rejection the residual w = max(0, p - q~_T) (w = p off
// the tail) with mass Zr = 1 - sum_tail min(p, q~_T) is used for recursive
// rejection of the remaining children, each a one-hot draft (accept with
// w(x)/Zr, else drop x); the bonus token is drawn from the final residual.
// p = softmax(t / T) over the whole vocabulary of the current node's target
// row (training-strategy paragraph: verification runs at temperature T).
//
// The walk is sequential in depth, so the latency of one level is what
// matters: every level's target row is split over the C CTAs of the tree's
// cluster (C and the CTA size chosen so that the whole batch fits in one
// wave with as many SMs per tree as that allows: the per-element exp2 of a
// slice runs at the SM's special-function rate).  Each warp of the cluster
// owns a contiguous slice of the row, loads all of it in one batch
// of predicated 16-byte loads (one memory latency per level) and keeps the
// slice's maximum and sum of exp2((t - max) * log2(e) / T) with packed
// float32x2 arithmetic.  Each warp stores its two numbers into the leader
// CTA's shared memory with asynchronous cluster stores that complete bytes of
// the leader's mbarrier (no fence on the sending side); no cluster-wide
// barrier is taken per level.  The leader forms the
// row normaliser, turns the target logits of the node's <= |S| support tokens
// (loaded at the start of the level, with the support itself prefetched when
// the previous level decided) into exact p, forms the residual in parallel and
// lets thread 0 take the <= K decisions, which reach the other CTAs the same
// way.  For the bonus token the slice masses locate
// the slice that holds it, and the leader reads only that slice again,
// scanning it in token-id order.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "st_common.cuh"
#include "st_kernels.h"

namespace cg = cooperative_groups;

namespace st {

constexpr int VER_MAX_THREADS = 1024;  // threads of a CTA: 256, 512 or 1024 (an SM runs 1024 at 64 registers)
constexpr int VER_WARPS = VER_MAX_THREADS / 32;
constexpr int VER_MAX_CLUSTER = 8;    // portable cluster size
constexpr int VER_WIDE_CLUSTER = 16;  // batches of <= num_sms / 16 trees with long rows: non-portable clusters
constexpr int VER_WIDE_MIN_V = 65536; //   of 16 CTAs, for rows of at least this many tokens
constexpr int VER_MAX_SLICES = VER_WARPS * VER_MAX_CLUSTER;
constexpr float LOG2E = 1.4426950408889634f;
constexpr double MASS_MARGIN = 1e-6;

struct VerShared {
  int32_t nd_parent[SPEC_TREE_MAX_NODES];      // leader: the tree's node arrays
  int32_t nd_slot[SPEC_TREE_MAX_NODES];
  int32_t nd_exp_row[SPEC_TREE_MAX_NODES];
  int32_t nd_token[SPEC_TREE_MAX_NODES];
  int32_t kid_by_slot[SPEC_TREE_MAX_SUPPORT];  // child node of each sibling slot, -1 if pruned
  float p_sup[SPEC_TREE_MAX_SUPPORT];          // p at support ranks of the node's draft row
  float qt_sup[SPEC_TREE_MAX_SUPPORT];         // q~_T at support ranks (0 off the tail)
  float w_sup[SPEC_TREE_MAX_SUPPORT];          // residual at support ranks
  float uv_lv[SPEC_TREE_MAX_SUPPORT];          // the level's accept uniforms, loaded at its start
  float all_m[2][VER_MAX_SLICES];              // leader, per level parity: every slice's maximum logit
  float all_s[2][VER_MAX_SLICES];              //   and sum of exp2((t - slice max) * c)
  uint64_t stats_bar[2];                       // leader: all slices of the level have arrived
  uint64_t dec_bar[2];                         // the leader's decision for the level has arrived
  int dec[2];                                  //   accepted child node, or -1
  float slice_corr[VER_MAX_SLICES];            // leader: per slice, sum over corrected tokens of (p - w)
  float red[VER_WARPS];
  int32_t corr_tok[SPEC_TREE_MAX_SUPPORT];     // corrected tokens inside the bonus slice
  float corr_w[SPEC_TREE_MAX_SUPPORT];
  float scan_w[VER_WARPS];
  int ncorr;
  float M;       // row maximum
  float invZp;   // 1 / sum of exp2((t - M) * c) over the row
  float Zr;      // residual mass
  int accepted;  // leader's decision of the level: accepted child node, or -1
  int nkids;     // children of the current node
  int bonus;
  int bonus_last;
  int bonus_slice;
  float bonus_target;  // target mass relative to the start of the bonus slice
  float u_bonus;       // the tree's bonus uniform, loaded at the start
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

// Slice g of ns: vectors [g * per, min((g + 1) * per, nvec)); the scalar tail
// (V not a multiple of the vector width) belongs to the last slice.
struct Slice {
  int v0, v1;
  __device__ Slice(int g, int ns, int nvec) {
    const int per = (nvec + ns - 1) / ns;
    v0 = min(g * per, nvec);
    v1 = min(v0 + per, nvec);
  }
};

__device__ __forceinline__ int slice_of_token(int v, int ns, int nvec, int vec) {
  const int per = (nvec + ns - 1) / ns;
  if (v >= nvec * vec || per == 0) return ns - 1;
  return min((v / vec) / per, ns - 1);
}

// ------------------------------------------------- packed float32x2 math ---
// Two IEEE float32 operations per instruction (round to nearest), so every
// result equals its scalar counterpart.
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rr;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rr, ra, rb;\n mov.b64 {%0, %1}, rr;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rr;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " sub.rn.f32x2 rr, ra, rb;\n mov.b64 {%0, %1}, rr;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rr;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rr, ra, rb;\n mov.b64 {%0, %1}, rr;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// The 16-byte vector as float pairs: element (2j, 2j+1) in pair j.
template <typename T>
struct Pairs;
template <>
struct Pairs<__nv_bfloat16> {
  static constexpr int N = 4;
  __device__ static __forceinline__ float2 get(const uint4& v, int j) {
    const uint32_t w = (j == 0) ? v.x : (j == 1) ? v.y : (j == 2) ? v.z : v.w;
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  __device__ static __forceinline__ uint4 neg_inf() { return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u); }
};
template <>
struct Pairs<float> {
  static constexpr int N = 2;
  __device__ static __forceinline__ float2 get(const uint4& v, int j) {
    return j == 0 ? make_float2(__uint_as_float(v.x), __uint_as_float(v.y))
                  : make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
  }
  __device__ static __forceinline__ uint4 neg_inf() { return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u); }
};

// Statistics of warp slice g of ns: maximum and sum of exp2((t - max) * c),
// c = log2(e) / T.  Every lane loads its vectors of the slice in batches of
// eight predicated 16-byte loads issued together (a 128K-token row split over
// 64 slices is one batch, so one memory latency); per batch the lane's
// running maximum is raised once, then each vector's elements contribute
// exp2((t - max) * c) in float pairs, and the vector sums enter a compensated
// per-lane sum.  Vectors holding NaN or +inf are left out and reported.
// Lanes combine in float32; lane 0 returns the slice's (max, sum).
template <typename T>
__device__ void slice_stats(const uint8_t* row, int V, int g, int ns, float c, bool& nonfinite, float& m_out,
                            float& s_out) {
  using E = VElem<T>;
  using P = Pairs<T>;
  constexpr int VEC = E::VEC;
  constexpr int BATCH = 8;
  const int lane = threadIdx.x & 31;
  const int nvec = static_cast<int>((static_cast<int64_t>(V) * E::ES) / 16);
  const Slice sl(g, ns, nvec);
  const uint4* rv = reinterpret_cast<const uint4*>(row);
  float m_run = -INFINITY;
  float2 s_run = make_float2(0.0f, 0.0f), comp = make_float2(0.0f, 0.0f);
  for (int base = sl.v0; base < sl.v1; base += 32 * BATCH) {
    uint4 v[BATCH];
#pragma unroll
    for (int k = 0; k < BATCH; ++k) {
      const int i = base + lane + 32 * k;
      v[k] = i < sl.v1 ? ldg_stream(rv + i) : P::neg_inf();
    }
    float bm = -INFINITY;
#pragma unroll
    for (int k = 0; k < BATCH; ++k) {
      const float vm = E::vmax(v[k]);
      if (!(vm < INFINITY)) {  // NaN or +inf: left out, reported
        nonfinite = true;
        v[k] = P::neg_inf();
      } else {
        bm = fmaxf(bm, vm);
      }
    }
    if (bm > m_run) {
      const float f = ex2((m_run - bm) * c);
      s_run = mul2(s_run, make_float2(f, f));
      comp = mul2(comp, make_float2(f, f));
      m_run = bm;
    }
    if (m_run == -INFINITY) continue;
    const float2 mm = make_float2(m_run, m_run), cc = make_float2(c, c);
#pragma unroll
    for (int k = 0; k < BATCH; ++k) {
      float2 vs = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int j = 0; j < P::N; ++j) {
        const float2 y = mul2(sub2(P::get(v[k], j), mm), cc);
        vs = add2(vs, make_float2(ex2(y.x), ex2(y.y)));
      }
      // compensated accumulation of the vector sums (pairwise lanes)
      const float2 yk = sub2(vs, comp);
      const float2 tk = add2(s_run, yk);
      comp = sub2(sub2(tk, s_run), yk);
      s_run = tk;
    }
  }
  float s_lane = (s_run.x - comp.x) + (s_run.y - comp.y);
  if (g == ns - 1) {
    const int tk = nvec * VEC + lane;
    if (tk < V) {
      const float x = E::load(row, tk);
      if (!(x < INFINITY)) nonfinite = true;
      if (x > -INFINITY && x < INFINITY) {
        if (x > m_run) {
          s_lane *= ex2((m_run - x) * c);
          m_run = x;
        }
        s_lane += ex2((x - m_run) * c);
      }
    }
  }
  float m = m_run;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
  float part = (m_run == -INFINITY) ? 0.0f : s_lane * ex2((m_run - m) * c);
  part = warp_sum(part);
  m_out = m;
  s_out = part;
}

// ------------------------------------------------- cluster signalling ---

__device__ __forceinline__ uint32_t cluster_addr(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}

// Asynchronous store of 4 bytes into the shared memory of a CTA of the
// cluster, completing 4 bytes of the transaction count of an mbarrier there
// (no fence: the data is visible to a thread that observes the phase).
__device__ __forceinline__ void st_async_b32(uint32_t addr, uint32_t v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr), "r"(v),
               "r"(bar)
               : "memory");
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

template <typename T, int C, int NT>
__global__ void __launch_bounds__(NT, VER_MAX_THREADS / NT) verify_kernel(VerifyLaunch L) {  // clusters of C CTAs
  using E = VElem<T>;
  constexpr int VEC = E::VEC;
  constexpr int NW = NT / 32;   // warps of a CTA
  constexpr int NS = NW * C;    // slices per row
  static_assert(NS <= VER_MAX_SLICES, "the slice statistics must fit the leader's arrays");
  extern __shared__ __align__(16) uint8_t smem_raw[];
  VerShared& s = *reinterpret_cast<VerShared*>(smem_raw);
  cg::cluster_group cluster = cg::this_cluster();
  const int cr = static_cast<int>(cluster.block_rank());
  const bool leader = cr == 0;
  const int b = blockIdx.x / C, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const spec_tree_t& t = L.tree;
  const int m = L.p.m, D = L.p.depth, K = L.p.K, S = L.S, V = L.V;
  const float Tmp = L.p.temperature;
  const float c = LOG2E / Tmp;
  const int64_t nb = static_cast<int64_t>(b) * t.max_nodes;
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.stats_bar[i], 1);  // the leader's expectation; the slices complete its bytes
      mbar_init(&s.dec_bar[i], 1);
    }
    fence_mbar_init();
  }
  // barriers initialised cluster-wide before any remote arrival (this needs
  // nothing from the previous kernel, so it overlaps that kernel's tail)
  cluster.sync();
  grid_dependency_wait();  // the tree comes from the previous kernel
  grid_dependents_launch();
  const int n_nodes = min(t.n_nodes[b], t.max_nodes);
  const int64_t row_bytes = L.row_stride * E::ES;
  const uint8_t* tgt = static_cast<const uint8_t*>(L.target);
  const int nvec = static_cast<int>((static_cast<int64_t>(V) * E::ES) / 16);
  if (leader) {
    // every entry of the node arrays (unused ones hold -1), so that these
    // loads need not wait for the node count
    const int nmax = min(t.max_nodes, SPEC_TREE_MAX_NODES);
    for (int i = tid; i < nmax; i += NT) {
      s.nd_parent[i] = t.node_parent[nb + i];
      s.nd_slot[i] = t.node_slot[nb + i];
      s.nd_exp_row[i] = t.node_exp_row[nb + i];
      s.nd_token[i] = t.node_token[nb + i];
    }
    if (tid == 0) s.u_bonus = L.u_bonus[b];
  }
  __syncthreads();  // the leader's node arrays
  bool nonfinite = false, timed_out = false;
  int node = 0, level = 0;
  int32_t* ot = L.out_tok + static_cast<int64_t>(b) * (D + 1);
  int32_t* on = L.out_node + static_cast<int64_t>(b) * (D + 1);
  // where this warp's slice statistics go in the leader's shared memory
  const uint32_t lead_m0 = cluster_addr(&s.all_m[0][cr * NW + warp], 0);
  const uint32_t lead_m1 = cluster_addr(&s.all_m[1][cr * NW + warp], 0);
  const uint32_t lead_s0 = cluster_addr(&s.all_s[0][cr * NW + warp], 0);
  const uint32_t lead_s1 = cluster_addr(&s.all_s[1][cr * NW + warp], 0);
  const uint32_t lead_bar0 = cluster_addr(&s.stats_bar[0], 0);
  const uint32_t lead_bar1 = cluster_addr(&s.stats_bar[1], 0);
  // support of the current node's draft row (leader): prefetched when the
  // previous level decided (for the root: now)
  int sup_v = -1, pp = -1;
  float sup_qt = 0.0f, zT = 0.0f;
  auto load_support = [&](int er) {
    if (er < 0) return;
    const int64_t srow = static_cast<int64_t>(b) * t.n_rows + er;
    if (tid < S) {
      sup_v = t.sup_id[srow * t.sup_stride + tid];
      sup_qt = t.sup_qT[srow * t.sup_stride + tid];
    }
    zT = t.sup_zT[srow];
    pp = t.probe_pos[srow];
  };
  if (leader) load_support(D > 0 ? s.nd_exp_row[0] : -1);
  while (true) {
    const int par = level & 1;
    const uint32_t wpar = static_cast<uint32_t>((level >> 1) & 1);
    const uint8_t* row = tgt + (nb + node) * row_bytes;
    const int er = leader && level < D ? s.nd_exp_row[node] : -1;
    // the level's accept uniforms, for thread 0's decisions after the barriers
    // below (its reads of the previous level's are done)
    if (er >= 0 && tid < K) s.uv_lv[tid] = L.u_verify[(static_cast<int64_t>(b) * D + level) * K + tid];
    // this level's expected bytes: every slice's two statistics (leader), the
    // decision (the others); a store may land before its expectation
    if (tid == 0) {
      if (leader) mbar_expect_tx(&s.stats_bar[par], static_cast<uint32_t>(NS) * 8u);
      else mbar_expect_tx(&s.dec_bar[par], 4u);
    }
    float wm, ws;
    slice_stats<T>(row, V, cr * NW + warp, NS, c, nonfinite, wm, ws);
    // target logits of the support tokens, landing while the slices arrive
    float t_sup = 0.0f;
    if (er >= 0 && tid < S) t_sup = E::load(row, sup_v);
    if (lane == 0) {
      const uint32_t bar = par ? lead_bar1 : lead_bar0;
      st_async_b32(par ? lead_m1 : lead_m0, __float_as_uint(wm), bar);
      st_async_b32(par ? lead_s1 : lead_s0, __float_as_uint(ws), bar);
    }
    int acc;
    if (leader) {
      if (!mbar_wait_cluster(&s.stats_bar[par], wpar)) timed_out = true;
      if (tid < K) s.kid_by_slot[tid] = -1;
      if (warp == 0) {
        // row maximum and normaliser (compensated per lane, pairwise across lanes)
        float mx = -INFINITY;
        for (int g = lane; g < NS; g += 32) mx = fmaxf(mx, s.all_m[par][g]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
        float z = 0.0f, zc = 0.0f;
        for (int g = lane; g < NS; g += 32) {
          const float am = s.all_m[par][g];
          const float x = am > -INFINITY ? s.all_s[par][g] * ex2((am - mx) * c) : 0.0f;
          const float y = x - zc;
          const float tt = z + y;
          zc = (tt - z) - y;
          z = tt;
        }
        z = warp_sum(z - zc);
        if (lane == 0) {
          s.M = mx;
          s.invZp = 1.0f / z;
          s.Zr = 1.0f;
          s.ncorr = 0;
        }
      }
      __syncthreads();
      // children of the node by sibling slot; a node at depth D is a leaf
      // (which also bounds the walk for malformed trees)
      if (er >= 0)
        for (int i = tid + 1; i < n_nodes; i += NT)
          if (s.nd_parent[i] == node) {
            const int slot = s.nd_slot[i];
            if (slot >= 0 && slot < K) s.kid_by_slot[slot] = i;
          }
      __syncthreads();
      int nk = 0;
      if (er >= 0)
        for (int k = 0; k < K; ++k) nk += s.kid_by_slot[k] >= 0;
      const float M = s.M, invZp = s.invZp;
      if (nk > 0) {
        const int probe_node = (pp >= 0 && m < K) ? s.kid_by_slot[m] : -1;
        const bool probe_last = L.p.verify_order == SPEC_TREE_PROBE_LAST;
        // probe first: the tail residual applies to the one-hot children iff the probe child survived
        const bool residual = probe_node >= 0 && !probe_last;
        float mn = 0.0f;
        if (tid < S) {
          const float p = expf(Tmp == 1.0f ? t_sup - M : (t_sup - M) / Tmp) * invZp;
          const float qt = (tid >= m && zT > 0.0f) ? sup_qt / zT : 0.0f;
          s.p_sup[tid] = p;
          s.qt_sup[tid] = qt;
          s.w_sup[tid] = (residual && tid >= m) ? fmaxf(0.0f, p - qt) : p;
          mn = (residual && tid >= m) ? fminf(p, qt) : 0.0f;
        }
        mn = warp_sum(mn);
        if (lane == 0) s.red[warp] = mn;
        __syncthreads();
        if (tid == 0) {
          const float* uv = s.uv_lv;
          int j = 0, accepted = -1;
          float Zr = 1.0f;
          bool empty = false;
          if (probe_node >= 0 && !probe_last) {
            const float p = s.p_sup[pp], qt = s.qt_sup[pp];
            const float u = uv[0];
            // near-tie: |u - ratio| < 1e-6 with ratio = p / q~_T
            if (L.margins && fabsf(u * qt - p) < static_cast<float>(MASS_MARGIN) * qt) atomicAdd(L.margins, 1u);
            if (u * qt < p) {
              accepted = probe_node;
            } else {
              float smin = 0.0f;
              for (int w = 0; w < (S + 31) / 32; ++w) smin += s.red[w];
              Zr = 1.0f - smin;
              j = 1;
            }
          }
          if (accepted < 0) {
            // one-hot children in slot order (the probe, if any, is done above or last)
            for (int slot = 0; slot < K; ++slot) {
              const int kid = s.kid_by_slot[slot];
              if (kid < 0 || kid == probe_node) continue;
              if (Zr <= 0.0f) {
                empty = true;
                break;
              }
              const int r = rank_of_slot(slot, m, pp);
              const float w = s.w_sup[r];
              const float u = uv[j];
              if (L.margins && fabsf(u * Zr - w) < static_cast<float>(MASS_MARGIN) * Zr) atomicAdd(L.margins, 1u);
              if (u * Zr < w) {
                accepted = kid;
                break;
              }
              Zr -= w;
              s.w_sup[r] = 0.0f;
              ++j;
            }
            if (probe_last && accepted < 0 && !empty && probe_node >= 0) {
              // the probe last, against the residual the one-hot rejections left
              if (Zr <= 0.0f) {
                empty = true;
              } else {
                const float w = s.w_sup[pp], qt = s.qt_sup[pp];
                const float u = uv[j];
                if (L.margins && fabsf(u * qt * Zr - w) < static_cast<float>(MASS_MARGIN) * qt * Zr)
                  atomicAdd(L.margins, 1u);
                if (u * qt * Zr < w) {
                  accepted = probe_node;
                } else {
                  // residual max(0, w - Zr q~_T) on the tail, of mass Zr - sum_tail min(w, Zr q~_T)
                  float smin = 0.0f;
                  for (int r = m; r < S; ++r) {
                    const float a = s.w_sup[r], q2 = Zr * s.qt_sup[r];
                    smin += fminf(a, q2);
                    s.w_sup[r] = fmaxf(0.0f, a - q2);
                  }
                  Zr -= smin;
                }
                ++j;
              }
            }
            if (accepted < 0 && !empty && Zr <= 0.0f) empty = true;
            if (empty) {
              // rounding emptied the residual: the bonus is drawn from p
              set_status(L.status, SPEC_TREE_S_RESIDUAL_EMPTY);
              for (int k = 0; k < S; ++k) s.w_sup[k] = s.p_sup[k];
              Zr = 1.0f;
            }
          }
          s.Zr = Zr;
          s.accepted = accepted;
          if (accepted >= 0) {
            ot[level] = s.nd_token[accepted];
            on[level] = accepted;
          }
        }
      } else if (tid == 0) {
        s.accepted = -1;
      }
      if (tid == 0) s.nkids = nk;
      __syncthreads();
      acc = s.accepted;
      // publish the decision to the other CTAs of the cluster
      if (tid >= 1 && tid < C)
        st_async_b32(cluster_addr(&s.dec[par], tid), static_cast<uint32_t>(acc), cluster_addr(&s.dec_bar[par], tid));
      // the next node's support, while the decision travels
      if (acc >= 0) load_support(level + 1 < D ? s.nd_exp_row[acc] : -1);
    } else {
      if (!mbar_wait_cluster(&s.dec_bar[par], wpar)) timed_out = true;
      acc = s.dec[par];
    }
    if (acc >= 0) {
      node = acc;
      ++level;
      continue;
    }
    if (!leader) break;  // the bonus is the leader's alone
    // ------------------------------------------------------------- bonus ---
    const int nk = s.nkids;
    const float M = s.M, invZp = s.invZp;
    for (int g = tid; g < NS; g += NT) s.slice_corr[g] = 0.0f;
    __syncthreads();
    const bool corrected = nk > 0 && tid < S && s.w_sup[tid] != s.p_sup[tid];
    if (corrected) atomicAdd(&s.slice_corr[slice_of_token(sup_v, NS, nvec, VEC)], s.p_sup[tid] - s.w_sup[tid]);
    __syncthreads();
    if (warp == 0) {
      // slice masses of w in id order; the first slice whose cumulative mass
      // exceeds u * Zr holds the bonus token
      constexpr int PER = (NS + 31) / 32;
      const float target = s.u_bonus * s.Zr;
      float mass[PER], run = 0.0f;
      int last_l = -1;
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int g = lane * PER + q;
        float x = 0.0f;
        if (g < NS) {
          const float am = s.all_m[level & 1][g];
          x = am > -INFINITY ? s.all_s[level & 1][g] * ex2((am - M) * c) * invZp : 0.0f;
          x -= s.slice_corr[g];
        }
        mass[q] = x;
        run += x;
        if (x > 0.0f) last_l = g;
      }
      float incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += y;
      }
      float acc_mass = incl - run;
      int pick = -1;
      float before = 0.0f;
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        if (pick < 0 && mass[q] > 0.0f && target < acc_mass + mass[q]) {
          pick = lane * PER + q;
          before = acc_mass;
        }
        acc_mass += mass[q];
      }
      const unsigned hit = __ballot_sync(FULL, pick >= 0);
      int bs;
      float bt;
      if (hit) {
        const int src = __ffs(hit) - 1;
        bs = __shfl_sync(FULL, pick, src);
        bt = target - __shfl_sync(FULL, before, src);
      } else {
        // rounding left the target past the total: the last slice with mass
        int lastg = last_l;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lastg = max(lastg, __shfl_xor_sync(FULL, lastg, o));
        bs = lastg < 0 ? NS - 1 : lastg;
        bt = 3.0e38f;
      }
      if (lane == 0) {
        s.bonus_slice = bs;
        s.bonus_target = bt;
        s.bonus = -1;
        s.bonus_last = -1;
      }
    }
    __syncthreads();
    const int bs = s.bonus_slice;
    const Slice sl(bs, NS, nvec);
    const int t0 = sl.v0 * VEC;
    const int t1 = (bs == NS - 1) ? V : sl.v1 * VEC;
    if (corrected && sup_v >= t0 && sup_v < t1) {
      const int k = atomicAdd(&s.ncorr, 1);
      s.corr_tok[k] = sup_v;
      s.corr_w[k] = s.w_sup[tid];
    }
    __syncthreads();
    // scan the slice in id order: thread i handles tokens [base + VEC * i, + VEC)
    {
      const int ncorr = s.ncorr;
      const float tr = s.bonus_target;
      const float tie = static_cast<float>(MASS_MARGIN) * s.Zr;  // a draw within 1e-6 * Zr of a boundary
      float base_run = 0.0f;
      int last_pos = -1;
      for (int cb = t0; cb < t1; cb += NT * VEC) {
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
          w[j] = (w[j] == -INFINITY) ? 0.0f : ex2((w[j] - M) * c) * invZp;
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
        for (int k = 0; k < NW; ++k) {
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
                if (L.margins && (tr - acc < tie || nx - tr < tie))
                  atomicAdd(L.margins + 1, 1u);
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
  if (timed_out) set_status(L.status, SPEC_TREE_S_TIMEOUT);
  // no CTA leaves while another may still write to its shared memory
  cluster.sync();
}

// Launch configuration of verify_kernel<T, C, NT>: the batch's clusters of
// C CTAs (a runtime cluster shape; above 8 CTAs a non-portable one),
// programmatic dependent launch on the stream.
template <typename T, int C, int NT>
cudaError_t verify_config(const VerifyLaunch& L, cudaStream_t stream, cudaLaunchConfig_t& cfg,
                          cudaLaunchAttribute (&attr)[2]) {
  const int smem = static_cast<int>(sizeof(VerShared));
  cudaError_t err = cudaFuncSetAttribute(verify_kernel<T, C, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err == cudaSuccess && C > VER_MAX_CLUSTER)
    err = cudaFuncSetAttribute(verify_kernel<T, C, NT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  cfg = cudaLaunchConfig_t{};
  cfg.gridDim = dim3(static_cast<unsigned>(L.B * C));
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return err;
}

template <typename T, int C, int NT>
cudaError_t launch_verify_c(const VerifyLaunch& L, cudaStream_t stream) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  cudaError_t err = verify_config<T, C, NT>(L, stream, cfg, attr);
  if (err != cudaSuccess) return err;
  return cudaLaunchKernelEx(&cfg, verify_kernel<T, C, NT>, L);
}

// Whether the device holds the batch's clusters of C CTAs in one wave.
template <typename T, int C, int NT>
bool verify_fits(const VerifyLaunch& L, cudaStream_t stream) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (verify_config<T, C, NT>(L, stream, cfg, attr) != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, verify_kernel<T, C, NT>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();  // the query's own error, not a launch's
    return false;
  }
  return n >= L.B;
}

template <typename T, int NT>
cudaError_t launch_verify_n(const VerifyLaunch& L, int C, cudaStream_t stream) {
  switch (C) {
    case 8:
      return launch_verify_c<T, 8, NT>(L, stream);
    case 4:
      return launch_verify_c<T, 4, NT>(L, stream);
    case 2:
      return launch_verify_c<T, 2, NT>(L, stream);
    default:
      return launch_verify_c<T, 1, NT>(L, stream);
  }
}

template <typename T>
cudaError_t launch_verify_t(const VerifyLaunch& L, cudaStream_t stream) {
  // Threads per tree: the most that keep the batch in one wave (an SM runs
  // 1024 threads at 64 registers), up to 8 CTAs of the smallest size that
  // gives one thread per support token (256 for |S| <= 256), spread over the
  // largest cluster (<= 8 CTAs).  More CTAs per tree put more SMs, and their
  // exp2 units, on the row of the slowest tree; small CTAs keep the leader's
  // per-level barriers cheap (at 1-16 trees, clusters of 8 CTAs of 256
  // threads beat clusters of 8 of 1024 by 5-11 us a step).  A cluster shape
  // the device cannot place is refused at launch, and the next smaller one is
  // tried.
  const int nt_min = L.S <= 256 ? 256 : L.S <= 512 ? 512 : VER_MAX_THREADS;
  // few trees with long rows: clusters of 16 CTAs of 256 threads (a level's
  // row summed on 16 SMs), when the device holds them all at once; shorter
  // rows leave too little work per CTA for the extra slices to pay
  if (nt_min == 256 && L.V >= VER_WIDE_MIN_V && static_cast<int64_t>(L.B) * VER_WIDE_CLUSTER <= L.num_sms &&
      verify_fits<T, VER_WIDE_CLUSTER, 256>(L, stream))
    return launch_verify_c<T, VER_WIDE_CLUSTER, 256>(L, stream);
  const int64_t budget = static_cast<int64_t>(L.num_sms) * VER_MAX_THREADS / L.B;
  int per_tree = VER_MAX_CLUSTER * nt_min;
  while (per_tree > nt_min && per_tree > budget) per_tree /= 2;
  cudaError_t err = cudaErrorInvalidValue;
  for (int C = min(VER_MAX_CLUSTER, per_tree / nt_min); C >= 1; C /= 2) {
    const int nt = max(nt_min, min(VER_MAX_THREADS, per_tree / C));
    err = nt == 256   ? launch_verify_n<T, 256>(L, C, stream)
          : nt == 512 ? launch_verify_n<T, 512>(L, C, stream)
                      : launch_verify_n<T, VER_MAX_THREADS>(L, C, stream);
    if (err == cudaSuccess) break;
  }
  return err;
}

cudaError_t launch_verify(const VerifyLaunch& L, cudaStream_t stream) {
  if (L.B == 0) return cudaSuccess;
  if (L.dtype == SPEC_TREE_BF16) return launch_verify_t<__nv_bfloat16>(L, stream);
  return launch_verify_t<float>(L, stream);
}

}  // namespace st
