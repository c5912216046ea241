// Launch descriptors shared by the host API and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "spec_tree.h"

namespace st {

struct SelLaunch {
  const void* logits;
  int64_t row_stride;  // elements
  int64_t in_rows;     // rows per tree in the logits and u_probe
  int64_t n_rows;      // rows per tree in the support arrays
  int64_t sup_row0;    // support row of a tree's first processed row
  int64_t rows_used;   // rows per tree to process
  int B, V, S, m;
  bool draw_probe;  // m < K: a probe child exists
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
  int num_sms;
  int ctas_per_sm;
  int32_t* sched;  // the tree's row counter (or NULL)
  bool dense;      // |S| = V > SPEC_TREE_MAX_SUPPORT: S is K, the ranks kept, plus the probe at entry K
};

struct RankLaunch {
  spec_tree_params p;
  int B, S;
  int64_t rows_avail;  // rows per tree that were expanded
  spec_tree_t tree;
  uint32_t* status;
  int probe_entry_cap;  // support entry of a probe of deeper rank: K for a dense support, else INT32_MAX
  // layer mode only
  int layer;
  void* state;
  int32_t* frontier_token;
  int32_t* frontier_parent;
};

struct VerifyLaunch {
  spec_tree_params p;
  int B, V, S, dtype;
  const void* target;
  int64_t row_stride;  // elements
  spec_tree_t tree;
  const float* u_verify;
  const float* u_bonus;
  int32_t* accept_len;
  int32_t* out_tok;
  int32_t* out_node;
  uint32_t* margins;
  uint32_t* status;
  int num_sms;
  // dense support: the draft rows the tree was built from
  const void* draft;
  int64_t draft_row_stride;  // elements
};

size_t select_expand_smem_bytes();
cudaError_t launch_select_expand(int dtype, const SelLaunch& L, cudaStream_t stream);
// supports of 129 to 1024 tokens
cudaError_t launch_select_wide(int dtype, const SelLaunch& L, cudaStream_t stream);
// batches with fewer rows than CTA slots: each row split over a cluster of
// select_split_parts(L) CTAs (1: no split, use the other kernels)
int select_split_parts(const SelLaunch& L);
cudaError_t launch_select_split(int dtype, const SelLaunch& L, cudaStream_t stream);
// the dense support of a vocabulary above SPEC_TREE_MAX_SUPPORT tokens
cudaError_t launch_select_dense(int dtype, const SelLaunch& L, cudaStream_t stream);
cudaError_t launch_rank_topr(const RankLaunch& L, cudaStream_t stream);
cudaError_t launch_rank_smart(const RankLaunch& L, cudaStream_t stream);
size_t layer_state_bytes();
cudaError_t launch_layer_topr(const RankLaunch& L, cudaStream_t stream);
cudaError_t launch_layer_finish(const RankLaunch& L, cudaStream_t stream);
cudaError_t launch_verify(const VerifyLaunch& L, cudaStream_t stream);
cudaError_t launch_verify_dense(const VerifyLaunch& L, cudaStream_t stream);

}  // namespace st
