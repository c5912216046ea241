// Host side of the C ABI (include/spec_tree.h): argument checks and launches.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "spec_tree.h"
#include "st_kernels.h"

namespace {

constexpr int MAX_DEVICES = 64;

int num_sms_of_current_device() {
  static int cache[MAX_DEVICES] = {0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

// |S| = min(support, V); support 0 selects the pages' default of 128 tokens
constexpr int DEFAULT_SUPPORT = 128;

int support_size(const spec_tree_params* p, int V) {
  if (p->support == SPEC_TREE_SUPPORT_DENSE) return V;
  const int s = p->support == 0 ? DEFAULT_SUPPORT : p->support;
  return s < V ? s : V;
}

// the dense support of a vocabulary too large for the support arrays
bool dense_support(const spec_tree_params* p, int V) {
  return p->support == SPEC_TREE_SUPPORT_DENSE && V > SPEC_TREE_MAX_SUPPORT;
}

// entries of a row's support arrays: |S|, or K + 1 for a dense support
int support_entries(const spec_tree_params* p, int V) {
  return dense_support(p, V) ? p->K + 1 : support_size(p, V);
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

int elem_size(int dtype) { return dtype == SPEC_TREE_BF16 ? 2 : (dtype == SPEC_TREE_F32 ? 4 : 0); }

int check_rows(int dtype, const void* logits, int64_t row_stride, int V) {
  const int es = elem_size(dtype);
  if (es == 0) return SPEC_TREE_E_LAYOUT;
  if (logits == nullptr) return SPEC_TREE_E_PARAM;
  if (row_stride < V) return SPEC_TREE_E_PARAM;
  if (!aligned16(logits) || (row_stride * es) % 16 != 0) return SPEC_TREE_E_LAYOUT;
  return SPEC_TREE_OK;
}

int check_tree(const spec_tree_params* p, const spec_tree_t* t, int V, bool need_nodes, bool need_sup) {
  if (t == nullptr) return SPEC_TREE_E_PARAM;
  const int S = support_entries(p, V);
  if (need_sup && (t->sup_id == nullptr || t->sup_q == nullptr || t->sup_qT == nullptr || t->sup_z == nullptr ||
                   t->sup_zT == nullptr || t->probe_pos == nullptr || t->sup_stride < S))
    return SPEC_TREE_E_PARAM;
  if (need_nodes && (t->node_token == nullptr || t->node_parent == nullptr || t->node_depth == nullptr ||
                     t->node_kind == nullptr || t->node_slot == nullptr || t->node_exp_row == nullptr ||
                     t->node_score == nullptr || t->n_nodes == nullptr || t->max_nodes < p->R + 1 ||
                     t->max_nodes > SPEC_TREE_MAX_NODES))
    return SPEC_TREE_E_PARAM;
  if (t->n_rows < spec_tree_rows_needed(p)) return SPEC_TREE_E_PARAM;
  return SPEC_TREE_OK;
}

cudaStream_t as_stream(spec_tree_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// bf16 rows of 8192 to 262144 tokens: the queue path's range
constexpr int SPLIT_MIN_V = 8192, SPLIT_MAX_V = 262144;

// the streaming kernel for supports of up to 128 tokens, else one CTA per row
// (the dense support of a large vocabulary by its own kernel); batches with
// fewer rows than CTA slots split each row over a cluster of CTAs
cudaError_t launch_select(int dtype, const st::SelLaunch& L, cudaStream_t stream) {
  if (L.dense) return st::launch_select_dense(dtype, L, stream);
  if (dtype == SPEC_TREE_BF16 && L.V >= SPLIT_MIN_V && L.V <= SPLIT_MAX_V && st::select_split_parts(L) > 1)
    return st::launch_select_split(dtype, L, stream);
  return L.S <= 128 ? st::launch_select_expand(dtype, L, stream) : st::launch_select_wide(dtype, L, stream);
}

// support entries the selection writes: |S|, or the K ranks kept of a dense support
void set_support(st::SelLaunch& L, const spec_tree_params* p, int V) {
  L.dense = dense_support(p, V);
  L.S = L.dense ? p->K : support_size(p, V);
}

int probe_entry_cap(const spec_tree_params* p, int V) { return dense_support(p, V) ? p->K : INT32_MAX; }

}  // namespace

extern "C" {

int spec_tree_rows_needed(const spec_tree_params* p) {
  if (p == nullptr) return 0;
  if (p->builder == SPEC_TREE_BUILDER_SMART) return p->R + 1;
  return 1 + (p->depth - 1) * p->W;
}

int spec_tree_check_params(const spec_tree_params* p, int V) {
  if (p == nullptr) return SPEC_TREE_E_PARAM;
  if (V < 1 || V >= (1 << 24)) return SPEC_TREE_E_PARAM;
  if (p->support < 0 || (p->support > SPEC_TREE_MAX_SUPPORT && p->support != SPEC_TREE_SUPPORT_DENSE))
    return SPEC_TREE_E_PARAM;
  const int S = support_size(p, V);
  if (p->K < 1 || p->K > S || p->m < 0 || p->m > p->K) return SPEC_TREE_E_PARAM;
  if (dense_support(p, V) && p->K > SPEC_TREE_DENSE_MAX_K) return SPEC_TREE_E_PARAM;
  if (p->verify_order != SPEC_TREE_PROBE_FIRST && p->verify_order != SPEC_TREE_PROBE_LAST) return SPEC_TREE_E_PARAM;
  if (p->depth < 1 || p->depth > 255 || p->R < 1 || p->R + 1 > SPEC_TREE_MAX_NODES) return SPEC_TREE_E_PARAM;
  if (!(p->temperature > 0.0f) || !isfinite(p->temperature)) return SPEC_TREE_E_PARAM;
  if (p->builder == SPEC_TREE_BUILDER_TOPR) {
    if (p->W < 1 || p->W > 4095 || p->W > SPEC_TREE_MAX_NODES) return SPEC_TREE_E_PARAM;
    const int64_t ncand = p->K + static_cast<int64_t>(p->depth - 1) * p->W * p->K;
    if (ncand > SPEC_TREE_MAX_CAND) return SPEC_TREE_E_PARAM;
  } else if (p->builder == SPEC_TREE_BUILDER_SMART) {
    if (static_cast<int64_t>(p->K) * (p->R + 1) > SPEC_TREE_MAX_CAND) return SPEC_TREE_E_PARAM;
    const float c[7] = {p->lambda, p->beta, p->gamma, p->delta, p->rho, p->eta, p->alpha};
    for (float x : c)
      if (!isfinite(x)) return SPEC_TREE_E_PARAM;
    if (p->lambda < 0.0f || p->gamma < 0.0f || p->delta < 0.0f || p->rho < 1.0f || !(p->alpha > 0.0f))
      return SPEC_TREE_E_PARAM;
  } else {
    return SPEC_TREE_E_PARAM;
  }
  return SPEC_TREE_OK;
}

int spec_tree_select_expand(const spec_tree_params* p, int B, int V, int dtype, const void* draft_logits,
                            int64_t row_stride, const float* u_probe, const spec_tree_t* tree, uint32_t* status,
                            spec_tree_stream_t stream) {
  int rc = spec_tree_check_params(p, V);
  if (rc) return rc;
  if (B < 0 || u_probe == nullptr) return SPEC_TREE_E_PARAM;
  if ((rc = check_rows(dtype, draft_logits, row_stride, V))) return rc;
  if ((rc = check_tree(p, tree, V, false, true))) return rc;
  const int needed = spec_tree_rows_needed(p);
  st::SelLaunch L;
  L.logits = draft_logits;
  L.row_stride = row_stride;
  L.in_rows = tree->n_rows;
  L.n_rows = tree->n_rows;
  L.sup_row0 = 0;
  L.rows_used = needed < tree->n_rows ? needed : tree->n_rows;
  L.B = B;
  L.V = V;
  set_support(L, p, V);
  L.m = p->m;
  L.draw_probe = p->m < p->K;
  L.temperature = p->temperature;
  L.u_probe = u_probe;
  L.sup_id = tree->sup_id;
  L.sup_q = tree->sup_q;
  L.sup_qT = tree->sup_qT;
  L.sup_z = tree->sup_z;
  L.sup_zT = tree->sup_zT;
  L.probe_pos = tree->probe_pos;
  L.sup_stride = tree->sup_stride;
  L.status = status;
  L.num_sms = num_sms_of_current_device();
  L.ctas_per_sm = 2;
  L.sched = tree->sched;
  if (L.num_sms <= 0) return SPEC_TREE_E_CUDA;
  return launch_select(dtype, L, as_stream(stream)) == cudaSuccess ? SPEC_TREE_OK : SPEC_TREE_E_CUDA;
}

int spec_tree_rank(const spec_tree_params* p, int B, int V, const spec_tree_t* tree, uint32_t* status,
                   spec_tree_stream_t stream) {
  int rc = spec_tree_check_params(p, V);
  if (rc) return rc;
  if (B < 0) return SPEC_TREE_E_PARAM;
  if ((rc = check_tree(p, tree, V, true, true))) return rc;
  st::RankLaunch L;
  L.p = *p;
  L.B = B;
  L.S = support_size(p, V);
  const int needed = spec_tree_rows_needed(p);
  L.rows_avail = needed < tree->n_rows ? needed : tree->n_rows;
  L.tree = *tree;
  L.status = status;
  L.probe_entry_cap = probe_entry_cap(p, V);
  L.layer = 0;
  L.state = nullptr;
  L.frontier_token = nullptr;
  L.frontier_parent = nullptr;
  const cudaError_t err = p->builder == SPEC_TREE_BUILDER_SMART ? st::launch_rank_smart(L, as_stream(stream))
                                                                 : st::launch_rank_topr(L, as_stream(stream));
  return err == cudaSuccess ? SPEC_TREE_OK : SPEC_TREE_E_CUDA;
}

int spec_tree_build(const spec_tree_params* p, int B, int V, int dtype, const void* draft_logits,
                    int64_t row_stride, const float* u_probe, const spec_tree_t* tree, uint32_t* status,
                    spec_tree_stream_t stream) {
  int rc = spec_tree_check_params(p, V);
  if (rc) return rc;
  if ((rc = check_tree(p, tree, V, true, true))) return rc;
  if ((rc = spec_tree_select_expand(p, B, V, dtype, draft_logits, row_stride, u_probe, tree, status, stream)))
    return rc;
  return spec_tree_rank(p, B, V, tree, status, stream);
}

size_t spec_tree_layer_state_bytes(void) { return st::layer_state_bytes(); }

int spec_tree_layer_rows(const spec_tree_params* p, int layer) {
  if (p == nullptr || p->builder != SPEC_TREE_BUILDER_TOPR || p->W < 1 || p->K < 1) return 0;
  if (layer < 0 || layer >= p->depth) return 0;
  if (layer == 0) return 1;
  int64_t ln = p->K;  // size of layer 1
  for (int d = 1; d < layer && ln <= SPEC_TREE_MAX_CAND; ++d) ln = (ln < p->W ? ln : p->W) * p->K;
  return static_cast<int>(ln < p->W ? ln : p->W);
}

int spec_tree_layer(const spec_tree_params* p, int B, int V, int layer, int dtype, const void* layer_logits,
                    int64_t row_stride, const float* u_probe, const spec_tree_t* tree, void* state,
                    int32_t* frontier_token, int32_t* frontier_parent, uint32_t* status,
                    spec_tree_stream_t stream) {
  int rc = spec_tree_check_params(p, V);
  if (rc) return rc;
  if (p->builder != SPEC_TREE_BUILDER_TOPR || layer < 0 || layer >= p->depth) return SPEC_TREE_E_PARAM;
  if (B < 0 || u_probe == nullptr || state == nullptr) return SPEC_TREE_E_PARAM;
  if (!aligned16(state)) return SPEC_TREE_E_LAYOUT;
  if ((rc = check_rows(dtype, layer_logits, row_stride, V))) return rc;
  if ((rc = check_tree(p, tree, V, false, true))) return rc;
  const int rows = spec_tree_layer_rows(p, layer);
  const int row0 = layer == 0 ? 0 : 1 + (layer - 1) * p->W;
  if (B == 0) return SPEC_TREE_OK;
  st::SelLaunch S;
  S.logits = layer_logits;
  S.row_stride = row_stride;
  S.in_rows = rows;
  S.n_rows = tree->n_rows;
  S.sup_row0 = row0;
  S.rows_used = rows;
  S.B = B;
  S.V = V;
  set_support(S, p, V);
  S.m = p->m;
  S.draw_probe = p->m < p->K;
  S.temperature = p->temperature;
  S.u_probe = u_probe;
  S.sup_id = tree->sup_id;
  S.sup_q = tree->sup_q;
  S.sup_qT = tree->sup_qT;
  S.sup_z = tree->sup_z;
  S.sup_zT = tree->sup_zT;
  S.probe_pos = tree->probe_pos;
  S.sup_stride = tree->sup_stride;
  S.status = status;
  S.num_sms = num_sms_of_current_device();
  S.ctas_per_sm = 2;
  S.sched = tree->sched;
  if (S.num_sms <= 0) return SPEC_TREE_E_CUDA;
  if (launch_select(dtype, S, as_stream(stream)) != cudaSuccess) return SPEC_TREE_E_CUDA;
  st::RankLaunch L;
  L.p = *p;
  L.B = B;
  L.S = support_size(p, V);
  L.rows_avail = rows;
  L.tree = *tree;
  L.status = status;
  L.probe_entry_cap = probe_entry_cap(p, V);
  L.layer = layer;
  L.state = state;
  L.frontier_token = frontier_token;
  L.frontier_parent = frontier_parent;
  return st::launch_layer_topr(L, as_stream(stream)) == cudaSuccess ? SPEC_TREE_OK : SPEC_TREE_E_CUDA;
}

int spec_tree_finish(const spec_tree_params* p, int B, int V, const spec_tree_t* tree, const void* state,
                     uint32_t* status, spec_tree_stream_t stream) {
  int rc = spec_tree_check_params(p, V);
  if (rc) return rc;
  if (p->builder != SPEC_TREE_BUILDER_TOPR || B < 0 || state == nullptr) return SPEC_TREE_E_PARAM;
  if (!aligned16(state)) return SPEC_TREE_E_LAYOUT;
  if ((rc = check_tree(p, tree, V, true, false))) return rc;
  st::RankLaunch L;
  L.p = *p;
  L.B = B;
  L.S = support_size(p, V);
  L.rows_avail = 0;
  L.tree = *tree;
  L.status = status;
  L.probe_entry_cap = probe_entry_cap(p, V);
  L.layer = p->depth;
  L.state = const_cast<void*>(state);
  L.frontier_token = nullptr;
  L.frontier_parent = nullptr;
  return st::launch_layer_finish(L, as_stream(stream)) == cudaSuccess ? SPEC_TREE_OK : SPEC_TREE_E_CUDA;
}

int spec_tree_verify(const spec_tree_params* p, int B, int V, int dtype, const void* target_logits,
                     int64_t row_stride, const spec_tree_t* tree, const float* u_verify, const float* u_bonus,
                     int32_t* accept_len, int32_t* out_tok, int32_t* out_node, uint32_t* margins, uint32_t* status,
                     spec_tree_stream_t stream) {
  int rc = spec_tree_check_params(p, V);
  if (rc) return rc;
  if (B < 0 || u_verify == nullptr || u_bonus == nullptr || accept_len == nullptr || out_tok == nullptr ||
      out_node == nullptr)
    return SPEC_TREE_E_PARAM;
  if (dense_support(p, V)) return SPEC_TREE_E_PARAM;  // spec_tree_verify_dense reads the draft rows too
  if ((rc = check_rows(dtype, target_logits, row_stride, V))) return rc;
  if ((rc = check_tree(p, tree, V, true, true))) return rc;
  st::VerifyLaunch L;
  L.p = *p;
  L.B = B;
  L.V = V;
  L.S = support_size(p, V);
  L.dtype = dtype;
  L.target = target_logits;
  L.row_stride = row_stride;
  L.tree = *tree;
  L.u_verify = u_verify;
  L.u_bonus = u_bonus;
  L.accept_len = accept_len;
  L.out_tok = out_tok;
  L.out_node = out_node;
  L.margins = margins;
  L.status = status;
  L.num_sms = num_sms_of_current_device();
  L.draft = nullptr;
  L.draft_row_stride = 0;
  if (L.num_sms <= 0) return SPEC_TREE_E_CUDA;
  return st::launch_verify(L, as_stream(stream)) == cudaSuccess ? SPEC_TREE_OK : SPEC_TREE_E_CUDA;
}

int spec_tree_verify_dense(const spec_tree_params* p, int B, int V, int dtype, const void* target_logits,
                           int64_t row_stride, const void* draft_logits, int64_t draft_row_stride,
                           const spec_tree_t* tree, const float* u_verify, const float* u_bonus,
                           int32_t* accept_len, int32_t* out_tok, int32_t* out_node, uint32_t* margins,
                           uint32_t* status, spec_tree_stream_t stream) {
  int rc = spec_tree_check_params(p, V);
  if (rc) return rc;
  if (!dense_support(p, V)) return SPEC_TREE_E_PARAM;
  if (B < 0 || u_verify == nullptr || u_bonus == nullptr || accept_len == nullptr || out_tok == nullptr ||
      out_node == nullptr)
    return SPEC_TREE_E_PARAM;
  if ((rc = check_rows(dtype, target_logits, row_stride, V))) return rc;
  if ((rc = check_rows(dtype, draft_logits, draft_row_stride, V))) return rc;
  if ((rc = check_tree(p, tree, V, true, true))) return rc;
  st::VerifyLaunch L;
  L.p = *p;
  L.B = B;
  L.V = V;
  L.S = V;
  L.dtype = dtype;
  L.target = target_logits;
  L.row_stride = row_stride;
  L.tree = *tree;
  L.u_verify = u_verify;
  L.u_bonus = u_bonus;
  L.accept_len = accept_len;
  L.out_tok = out_tok;
  L.out_node = out_node;
  L.margins = margins;
  L.status = status;
  L.num_sms = num_sms_of_current_device();
  L.draft = draft_logits;
  L.draft_row_stride = draft_row_stride;
  if (L.num_sms <= 0) return SPEC_TREE_E_CUDA;
  return st::launch_verify_dense(L, as_stream(stream)) == cudaSuccess ? SPEC_TREE_OK : SPEC_TREE_E_CUDA;
}

const char* spec_tree_strerror(int code) {
  switch (code) {
    case SPEC_TREE_OK:
      return "ok";
    case SPEC_TREE_E_PARAM:
      return "invalid parameter or null pointer";
    case SPEC_TREE_E_LAYOUT:
      return "unsupported dtype or rows not 16-byte aligned";
    case SPEC_TREE_E_CUDA:
      return "CUDA launch failed";
    default:
      return "unknown error";
  }
}

}  // extern "C"
