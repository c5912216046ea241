// The expansion epilogue of a support of up to 128 tokens, by one warp:
// shared by the streaming kernel's selector warp and the leader CTA of the
// split-row kernel, so that both give bit-identical supports.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "st_common.cuh"
#include "st_keys.cuh"

namespace st {

// Softmaxes, tail masses and the probe of one row from its sorted support,
// by the selector warp (rank j*32 + lane in val[j]).  RheoSampling Key design
// 2; the probe is the first tail rank k with u * z_T < sum_{j=m..k} q_T(j),
// computed on unnormalised weights.
template <typename T, typename A>
__device__ void expand_epilogue(const uint64_t (&val)[4], const A& a, int64_t out_row, int64_t in_row, int n_sup) {
  const int lane = threadIdx.x & 31;
  float l[4], e[4], eT[4];
  const float lmax = key_value<T>(static_cast<uint32_t>(__shfl_sync(FULL, val[0], 0) >> 32));
  if (lane == 0 && !(lmax < INFINITY)) set_status(a.status, SPEC_TREE_S_NONFINITE_DRAFT);
  const bool unit_T = a.temperature == 1.0f;  // then the tempered weights are the untempered ones
  float se = 0.0f, seT = 0.0f, te = 0.0f, teT = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = j * 32 + lane;
    const bool valid = r < n_sup;
    l[j] = key_value<T>(static_cast<uint32_t>(val[j] >> 32));
    const float dd = l[j] - lmax;
    e[j] = valid ? expf(dd) : 0.0f;
    eT[j] = unit_T ? e[j] : (valid ? expf(dd / a.temperature) : 0.0f);
    se += e[j];
    seT += eT[j];
    if (valid && r >= a.m) {
      te += e[j];
      teT += eT[j];
    }
  }
  // the four sums, their butterfly steps interleaved
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    se += __shfl_xor_sync(FULL, se, o);
    seT += __shfl_xor_sync(FULL, seT, o);
    te += __shfl_xor_sync(FULL, te, o);
    teT += __shfl_xor_sync(FULL, teT, o);
  }
  int32_t* sid = a.sup_id + out_row * a.sup_stride;
  float* sq = a.sup_q + out_row * a.sup_stride;
  float* sqT = a.sup_qT + out_row * a.sup_stride;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = j * 32 + lane;
    if (r < n_sup) {
      sid[r] = static_cast<int32_t>(~static_cast<uint32_t>(val[j]));
      sq[r] = e[j] / se;
      sqT[r] = eT[j] / seT;
    }
  }
  int probe = -1;
  if (a.draw_probe && a.m < n_sup && teT > 0.0f) {
    // inclusive scans of the tempered tail weights of the four rank blocks,
    // interleaved, then the blocks' carries
    const float target = a.u_probe[in_row] * teT;
    float x[4], incl[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = j * 32 + lane;
      x[j] = (r < n_sup && r >= a.m) ? eT[j] : 0.0f;
      incl[j] = x[j];
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float y = __shfl_up_sync(FULL, incl[j], o);
        if (lane >= o) incl[j] += y;
      }
    }
    float carry = 0.0f;
    int last = -1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = j * 32 + lane;
      const bool tl = r < n_sup && r >= a.m;
      const unsigned hit = __ballot_sync(FULL, tl && target < carry + incl[j]);
      if (probe < 0 && hit) probe = j * 32 + __ffs(hit) - 1;
      const unsigned pos = __ballot_sync(FULL, tl && x[j] > 0.0f);
      if (pos) last = j * 32 + 31 - __clz(pos);
      carry += __shfl_sync(FULL, incl[j], 31);
    }
    if (probe < 0) probe = last;
  }
  if (lane == 0) {
    a.sup_z[out_row] = te / se;
    a.sup_zT[out_row] = teT / seT;
    a.probe_pos[out_row] = probe;
  }
}

}  // namespace st
