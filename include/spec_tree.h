/*
 * spec_tree.h -- C ABI of the GB300 (sm_103a) hot path of stochastic
 * dynamic-tree speculative decoding.
 *
 * Sources of the operations (papernotes.org pages):
 *   "RheoSampling: Resolving the One-Hot Dilemma in Stochastic Dynamic-Tree
 *    Speculative Decoding" (NeurIPS 2026 notes), Method:
 *     - Key design 1: top-128 truncation of the draft logits before the softmax;
 *     - Key design 2: dual-identity expansion (top-m deterministic children, one
 *       probe from the renormalised tail with proxy probability min{q(x_m), z},
 *       fillers) and the Local Ranking Preservation lemma;
 *     - overall framework / flowchart: cumulative path scores, global top-R pruning;
 *     - Key design 3: optimal-transport verification (probe first, residual
 *       norm(max(0, p - q~)), recursive rejection, bonus token);
 *     - training-strategy paragraph: build/prune on untempered draft
 *       probabilities, sample the probe and verify at temperature T.
 *   "SMART: When is it Actually Worth Expanding a Speculative Tree?" (ECCV 2026
 *    notes), Method / Key designs 1-3: the marginal keep rule with the cost
 *    models lambda*|T| + beta and gamma*(exp(delta*|T|^rho) - 1) + eta.
 *
 * General contract of every entry point:
 *   - Pointers named "device" are device pointers owned by the caller; the
 *     library allocates nothing, keeps no state between calls (except
 *     spec_tree_layer_static, whose state lives in the library) and never
 *     synchronises the host.  Every call is asynchronous on `stream`
 *     (0 = the legacy default stream).
 *   - Return value: SPEC_TREE_OK (0) or a negative SPEC_TREE_E_* code.
 *     Argument errors are detected on the host before any launch, so nothing
 *     has been enqueued when a call returns SPEC_TREE_E_PARAM or
 *     SPEC_TREE_E_LAYOUT.  SPEC_TREE_E_CUDA reports a failed launch.
 *   - Anomalies only the device can see (a NaN or +inf logit, an empty
 *     residual after rounding, a bounded wait that gave up) are OR-ed into the
 *     caller's device word `status` (SPEC_TREE_S_* bits).  Kernels never trap
 *     and every wait is bounded.  The caller zeroes `status` when it wants a
 *     fresh reading.
 *   - Logit rows are row-major with `row_stride` elements between rows; a
 *     row starts on a 16-byte boundary (base pointer 16-byte aligned and
 *     row_stride * element size a multiple of 16), else SPEC_TREE_E_LAYOUT.
 *     V need not be a multiple of 8.
 */
#ifndef SPEC_TREE_H
#define SPEC_TREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA runtime header. */
typedef struct CUstream_st* spec_tree_stream_t;

/* element types of logit rows */
#define SPEC_TREE_BF16 0
#define SPEC_TREE_F32 1

/* tree builders */
#define SPEC_TREE_BUILDER_TOPR 0  /* expand-then-rerank, frontier top-W, global top-R */
#define SPEC_TREE_BUILDER_SMART 1 /* SMART marginal keep rule, budget R */

/* verification orders */
#define SPEC_TREE_PROBE_FIRST 0
#define SPEC_TREE_PROBE_LAST 1

/* node kinds */
#define SPEC_TREE_ROOT 0
#define SPEC_TREE_DET 1
#define SPEC_TREE_PROBE 2
#define SPEC_TREE_FILL 3

/* return codes */
#define SPEC_TREE_OK 0
#define SPEC_TREE_E_PARAM (-1)  /* bad parameter or null pointer */
#define SPEC_TREE_E_LAYOUT (-3) /* unsupported dtype or misaligned rows */
#define SPEC_TREE_E_CUDA (-4)   /* a kernel launch failed */

/* device status bits */
#define SPEC_TREE_S_NONFINITE_DRAFT 1u   /* NaN or +inf in a draft row read */
#define SPEC_TREE_S_NONFINITE_TARGET 2u  /* NaN or +inf in a target row read */
#define SPEC_TREE_S_RESIDUAL_EMPTY 4u    /* residual mass <= 0 after rounding; bonus drawn from p */
#define SPEC_TREE_S_OVERFLOW 8u          /* internal candidate buffer overflow (not expected) */
#define SPEC_TREE_S_TIMEOUT 16u          /* a bounded wait on a bulk copy gave up */
#define SPEC_TREE_S_ROWS 32u             /* a tree wanted more draft rows than n_rows */
#define SPEC_TREE_S_LAYERS 64u           /* layer mode: a call out of order, or finish before the last layer */

/* Limits of this build. */
#define SPEC_TREE_MAX_SUPPORT 1024
/* support = SPEC_TREE_SUPPORT_DENSE: |S| = V, the whole vocabulary (the
 * pages' "full dense" support).  Above SPEC_TREE_MAX_SUPPORT tokens the
 * support arrays keep only ranks 0..K-1 and the probe (see spec_tree_t), K is
 * at most SPEC_TREE_DENSE_MAX_K, and verification takes the draft rows too
 * (spec_tree_verify_dense). */
#define SPEC_TREE_SUPPORT_DENSE 0x40000000
#define SPEC_TREE_DENSE_MAX_K 64
#define SPEC_TREE_MAX_CAND 2048 /* K + (depth-1)*W*K for the top-R builder; K*R for SMART */
#define SPEC_TREE_MAX_NODES 512 /* R + 1 */

/*
 * Parameters of the method.
 *   K        children (slots) per expanded node, 1 <= K <= support.
 *   m        deterministic children (top-m), 0 <= m <= K.  m = K gives the
 *            one-hot Top-K tree (every child deterministic, no probe): the
 *            pages' Top-K baseline.
 *   W        frontier width: nodes expanded per layer (top-R builder).
 *   depth    D >= 1: layers of draft nodes.
 *   R        pruned tree size in draft nodes, root excluded (top-R builder);
 *            node budget (SMART).  Node arrays hold R + 1 entries.
 *   support  |S| = min(support, V); 0 means 128.  1 <= support <= 1024 (the
 *            pages' ablation: 128, 256, 512, 1024; support >= V is the dense
 *            support of a vocabulary of at most 1024 tokens), or
 *            SPEC_TREE_SUPPORT_DENSE: |S| = V for any vocabulary.
 *   temperature T > 0: probe sampling and verification use q_T and
 *            p = softmax(t / T); ranking uses untempered q.
 *   builder  SPEC_TREE_BUILDER_TOPR or SPEC_TREE_BUILDER_SMART.
 *   lambda, beta, gamma, delta, rho, eta, alpha: SMART cost model (units of
 *            one target decoding step) and discount; ignored by top-R.
 *   verify_order SPEC_TREE_PROBE_FIRST: the probe is tested first and the
 *            others are one-hot drafts under its residual (RheoSampling Key
 *            design 3, optimal-transport verification); SPEC_TREE_PROBE_LAST:
 *            the one-hot children first, the probe last against the residual
 *            they leave (recursive rejection sampling with the probe as one
 *            more draft, the pages' "Rheo + RRSw" ablation).
 */
typedef struct spec_tree_params {
  int32_t K, m, W, depth, R, support;
  float temperature;
  int32_t builder;
  float lambda, beta, gamma, delta, rho, eta, alpha;
  int32_t verify_order;
} spec_tree_params;

/*
 * Tree buffers (all device pointers, caller-owned).  B trees; `n_rows` draft
 * rows and `max_nodes` (= R + 1) node entries per tree.
 *
 * Node arrays [B][max_nodes], canonical order: node 0 is the root, then depth
 * ascending, then ranking key (score descending, creation index ascending).
 * Entries at index >= n_nodes[b] hold token/parent/exp_row = -1, score 0.
 *   node_token   token id (root: -1)
 *   node_parent  index of the parent node (root: -1)
 *   node_depth   0 for the root
 *   node_kind    SPEC_TREE_ROOT/DET/PROBE/FILL
 *   node_slot    sibling slot (DET 0..m-1, PROBE m, FILL after; root -1)
 *   node_exp_row draft row the node was expanded from, -1 if not expanded
 *   node_score   cumulative path score (the probe contributes its proxy)
 *   n_nodes      [B] node count including the root
 * Support arrays, per draft row [B][n_rows] (support ranks 0..|S|-1):
 *   sup_id [.][S] token ids by (logit desc, id asc); sup_q / sup_qT [.][S]
 *   untempered / tempered truncated softmax; sup_z / sup_zT tail masses over
 *   ranks m..|S|-1; probe_pos rank of the probe in S (-1: no probe).
 *   `sup_stride` is the per-row capacity of sup_id/sup_q/sup_qT (>= |S|).
 *   Dense support of V > SPEC_TREE_MAX_SUPPORT tokens: entries 0..K-1 hold
 *   support ranks 0..K-1 (all children but the probe come from there) and
 *   entry K the probe (its id, q and q_T; probe_pos is still its rank in the
 *   whole vocabulary), so sup_stride >= K + 1; q, q_T and the tail masses are
 *   over the whole vocabulary.
 * Row schedule (optional, may be NULL):
 *   sched        device uint32[3], zero before the first call that uses it.
 *                [0], [1]: the support selection hands draft rows to its CTAs
 *                on demand from this counter (a CTA that runs ahead takes
 *                more rows, so they finish together) and leaves both words at
 *                zero again when it ends.  [2]: the top-|S| cut key of a
 *                recent row (of the latest call, or of the latest row finished
 *                when rows are selected one CTA or one cluster per row, which
 *                rows starting later in the same call read too), taken as the
 *                predicted queue threshold of the next rows (a hint only: a
 *                wrong value costs time, never a different result; any value
 *                is valid).  NULL: rows are dealt to the CTAs in a fixed
 *                order, no hint is kept.
 *                Calls that overlap on the GPU must not share one counter.
 */
typedef struct spec_tree_t {
  int32_t* node_token;
  int32_t* node_parent;
  int32_t* node_depth;
  int32_t* node_kind;
  int32_t* node_slot;
  int32_t* node_exp_row;
  float* node_score;
  int32_t* n_nodes;
  int32_t* sup_id;
  float* sup_q;
  float* sup_qT;
  float* sup_z;
  float* sup_zT;
  int32_t* probe_pos;
  int32_t n_rows;
  int32_t max_nodes;
  int32_t sup_stride;
  int32_t* sched;
} spec_tree_t;

/* Draft rows one tree consumes: 1 + (depth-1)*W (top-R), at most R + 1 (SMART). */
int spec_tree_rows_needed(const spec_tree_params* p);

/* Host-only check of the parameters against vocabulary size V (no CUDA call). */
int spec_tree_check_params(const spec_tree_params* p, int V);

/*
 * Support selection and dual-identity expansion of every draft row
 * (RheoSampling Key designs 1-2).  For each tree b and row e < rows, where
 * rows = min(tree->n_rows, spec_tree_rows_needed(p)):
 *   S = top-|S| token ids of draft row (b, e) by (logit desc, id asc);
 *   q, q_T = softmax over S of l and of l / T (untempered / tempered);
 *   z, z_T = their sums over ranks m..|S|-1 (the tail);
 *   probe = first tail rank k, in rank order, with
 *           u_probe[b][e] * z_T < sum_{j=m..k} q_T(j)   (none if z_T == 0).
 * draft_logits: device [B][tree->n_rows][row_stride] of dtype (bf16 or f32).
 * u_probe:      device [B][tree->n_rows] float, U[0,1).
 * Writes the sup_* arrays and probe_pos of `tree`.
 */
int spec_tree_select_expand(const spec_tree_params* p, int B, int V, int dtype,
                            const void* draft_logits, int64_t row_stride,
                            const float* u_probe, const spec_tree_t* tree,
                            uint32_t* status, spec_tree_stream_t stream);

/*
 * Tree building from the expanded rows (RheoSampling overall framework:
 * path scores, frontier top-W per layer, global top-R; or SMART Key design 3
 * keep rule).  Reads the sup_* arrays written by spec_tree_select_expand and
 * writes the node arrays and n_nodes.  Child scores are fl(parent x q) in
 * float32 (parent x proxy for the probe); the ranking key never involves a
 * token id, so a probe's survival does not depend on its identity.
 */
int spec_tree_rank(const spec_tree_params* p, int B, int V, const spec_tree_t* tree,
                   uint32_t* status, spec_tree_stream_t stream);

/* spec_tree_select_expand followed by spec_tree_rank on the same stream. */
int spec_tree_build(const spec_tree_params* p, int B, int V, int dtype,
                    const void* draft_logits, int64_t row_stride,
                    const float* u_probe, const spec_tree_t* tree,
                    uint32_t* status, spec_tree_stream_t stream);

/*
 * Layer-by-layer verification of built trees (RheoSampling Key design 3).
 * For each tree, from the root: p = softmax(t / T) over the full vocabulary
 * of the current node's target row.  With SPEC_TREE_PROBE_FIRST the node's
 * children are tested probe first (accept iff u < p(x_s) / q~_T(x_s)), then,
 * under the residual w = max(0, p - q~_T) on the tail (w = p elsewhere, mass
 * Zr = 1 - sum_tail min(p, q~_T)), each remaining child x in slot order
 * (accept iff u < w(x) / Zr, else Zr -= w(x), w(x) = 0).  Without a probe
 * child, w = p and Zr = 1.  With SPEC_TREE_PROBE_LAST the children other
 * than the probe go first under w = p, Zr = 1 (as above), then the probe is
 * accepted iff u < (w(x_s) / Zr) / q~_T(x_s), and on rejection the residual
 * becomes max(0, w - Zr q~_T), of mass Zr - sum_tail min(w, Zr q~_T).  The j-th decision at level l uses
 * u_verify[b][l][j].  An accepted child becomes the node; when every child
 * is rejected or the node has none, the bonus token is the first token in id
 * order with u_bonus[b] * Zr < sum_{v' <= v} w(v').
 *   target_logits: [B][tree->max_nodes][row_stride]; row i is the target
 *                  logits at node i.  Only rows on the accepted path are
 *                  read, with plain loads, so the array may also live in
 *                  pinned host memory (cudaHostAlloc; its host pointer is a
 *                  valid device address under unified addressing): the
 *                  kernel then reads just those rows over NVLink-C2C (or
 *                  PCIe) instead of the caller copying every row to HBM.
 *   u_verify: device [B][depth][K] float; u_bonus: device [B] float.
 *   accept_len: device [B]; out_tok, out_node: device [B][depth + 1]
 *   (accepted tokens then the bonus token; accepted node indices then -1;
 *   unused entries -1).
 *   margins: device uint32[2] or NULL; counts near-tie decisions, whose
 *   float32 outcome could differ from an exact computation: [0] accept tests
 *   with |u - ratio| < 1e-6 (ratio = the accept probability before the
 *   min(1, .)), [1] bonus draws whose target u * Zr lies within 1e-6 * Zr of
 *   a boundary of the residual's cumulative mass.  Added to, never cleared.
 */
int spec_tree_verify(const spec_tree_params* p, int B, int V, int dtype,
                     const void* target_logits, int64_t row_stride,
                     const spec_tree_t* tree, const float* u_verify, const float* u_bonus,
                     int32_t* accept_len, int32_t* out_tok, int32_t* out_node,
                     uint32_t* margins, uint32_t* status, spec_tree_stream_t stream);

/*
 * spec_tree_verify for a tree built on the dense support of a vocabulary of
 * more than SPEC_TREE_MAX_SUPPORT tokens (support = SPEC_TREE_SUPPORT_DENSE;
 * RheoSampling notes, Key design 3 with Key design 1's dense support).  The
 * tail law q~_T(v) = q_T(v) / z_T then covers every token but the m
 * deterministic ones, and the tree's support arrays keep only its first
 * ranks, so the kernel recomputes q_T(v) = exp((d_v - d_max) / T) q_T(x_1)
 * from the node's draft row d (d_max its rank-0 logit): the residual mass
 * 1 - sum_tail min(p, q~_T) and the bonus then take a pass over the target
 * and the draft row of the node.
 *   draft_logits: the draft rows the tree was built from, [B][tree->n_rows]
 *                 [draft_row_stride] of dtype, 16-byte aligned rows; only the
 *                 rows of accepted-path nodes whose probe was rejected are read.
 * Everything else is as for spec_tree_verify.  Returns SPEC_TREE_E_PARAM for
 * a tree whose support is not dense, or V <= SPEC_TREE_MAX_SUPPORT (where
 * spec_tree_verify handles the dense support).
 */
int spec_tree_verify_dense(const spec_tree_params* p, int B, int V, int dtype,
                           const void* target_logits, int64_t row_stride,
                           const void* draft_logits, int64_t draft_row_stride,
                           const spec_tree_t* tree, const float* u_verify, const float* u_bonus,
                           int32_t* accept_len, int32_t* out_tok, int32_t* out_node,
                           uint32_t* margins, uint32_t* status, spec_tree_stream_t stream);

/*
 * Layer mode: the top-R tree of spec_tree_build, built one layer per call so
 * that the draft model can run on each frontier in between (RheoSampling
 * overall framework: the frontier is expanded layer by layer).  Top-R builder
 * only (SPEC_TREE_BUILDER_SMART returns SPEC_TREE_E_PARAM).
 *
 * For layer = 0, 1, ..., depth - 1 in order, per batch of trees:
 *   spec_tree_layer(layer): expands the rows_l = spec_tree_layer_rows(p, layer)
 *     draft rows of the current frontier (layer 0: the root) exactly as
 *     spec_tree_select_expand does, into support rows r0 .. r0 + rows_l - 1 of
 *     `tree` (r0 = 0 for layer 0, else 1 + (layer - 1) * W), scores their
 *     children (the candidates of depth layer + 1), ranks them in their
 *     layer and, unless layer = depth - 1, names the next frontier: its first
 *     W candidates by key.
 *       layer_logits: device [B][rows_l][row_stride] of dtype; row f holds the
 *         draft logits after frontier rank f of the previous call's frontier
 *         (layer 0: after the root).
 *       u_probe: device [B][rows_l] float, U[0,1): row f's probe draw.
 *       state: device, B * spec_tree_layer_state_bytes() bytes, 16-byte
 *         aligned, owned by the caller; written by layer 0, read and updated
 *         by every later call, read by spec_tree_finish.  No initialisation
 *         is needed.
 *       frontier_token, frontier_parent: device [B][W] int32, or NULL: the
 *         token of frontier rank f (the draft's next input for row f of the
 *         next call) and the previous frontier's rank of its parent (-1 for
 *         the root's children); -1 past the frontier and after the last layer.
 *   spec_tree_finish: the global top-R cut; writes the node arrays and
 *     n_nodes of `tree`, equal to what spec_tree_build writes for the same
 *     draft rows and draws.
 * A call out of order sets SPEC_TREE_S_LAYERS and spoils the tree's state
 * until the next layer 0; spec_tree_finish then writes the root alone.
 */
size_t spec_tree_layer_state_bytes(void);

/* Frontier rows expanded by call `layer` (host only): 1 for layer 0, else
 * min(W, size of layer `layer`); 0 if layer is out of range or p invalid. */
int spec_tree_layer_rows(const spec_tree_params* p, int layer);

int spec_tree_layer(const spec_tree_params* p, int B, int V, int layer, int dtype,
                    const void* layer_logits, int64_t row_stride, const float* u_probe,
                    const spec_tree_t* tree, void* state, int32_t* frontier_token,
                    int32_t* frontier_parent, uint32_t* status, spec_tree_stream_t stream);

int spec_tree_finish(const spec_tree_params* p, int B, int V, const spec_tree_t* tree,
                     const void* state, uint32_t* status, spec_tree_stream_t stream);

/*
 * spec_tree_layer_static: spec_tree_layer for callers that cannot allocate
 * device memory.  The pages have no counterpart: this is an interface
 * variant of the layer-by-layer builder, not a step of the method.
 *
 * Who needs it: a draft loop embedded in a host runtime that reserves all
 * device memory up front and gives its plugins no allocator, and decode
 * loops that must not call cudaMalloc or cudaFree because those can
 * synchronise the device in the middle of a step.  Such a caller still owns
 * the logits, draws, tree and frontier buffers, but cannot provide the
 * builder's per-tree state (spec_tree_layer_state_bytes() per tree).
 *
 * What differs from spec_tree_layer:
 *   - the state lives in a device array inside this library, sized for
 *     SPEC_TREE_STATIC_MAX_TREES trees (3.5 MiB, held on every GPU that loads
 *     the library until the process exits); B > SPEC_TREE_STATIC_MAX_TREES
 *     returns SPEC_TREE_E_PARAM before anything is launched;
 *   - the call of the last layer (layer = depth - 1) also performs
 *     spec_tree_finish, so it writes the node arrays and n_nodes of `tree`
 *     (its arguments are checked before the first launch);
 *   - the array is shared by every call in the process and keeps the last
 *     call's contents.  Layer 0 rewrites everything later calls read, so
 *     nothing needs clearing, but two builds whose calls overlap on the GPU
 *     (on different streams, or from different host threads) race on it:
 *     finish one batch's layers before another batch's layer 0 starts;
 *   - the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.  A failed lookup returns
 *     SPEC_TREE_E_CUDA.  The cached address belongs to the device's primary
 *     context at that first call: a cudaDeviceReset of that device afterwards
 *     (which unloads the library's module and may place the array elsewhere
 *     when it is loaded again) is not supported by this entry point.
 * It calls no cudaMalloc, cudaFree or other allocating routine.  Everything
 * else (arguments, rows, frontier outputs, status bits, results bit for bit)
 * is as for spec_tree_layer followed, after the last layer, by
 * spec_tree_finish.
 */
#define SPEC_TREE_STATIC_MAX_TREES 64

int spec_tree_layer_static(const spec_tree_params* p, int B, int V, int layer, int dtype,
                           const void* layer_logits, int64_t row_stride, const float* u_probe,
                           const spec_tree_t* tree, int32_t* frontier_token, int32_t* frontier_parent,
                           uint32_t* status, spec_tree_stream_t stream);

/*
 * SMART cost-model fit from profiled steps (SMART notes, Key design 2:
 * device profiling, least squares over a few forward passes, the biases
 * fixed at zero so that both curves pass through the origin).  Host only, no
 * CUDA call.
 *   n[i] > 0:        tree size (tokens) of profiled step i, i < npts, 3 <= npts <= 1024;
 *   t_draft[i] >= 0: its drafting time;  t_verify[i] >= 0: its verification time;
 *   t_base > 0:      the time of a plain target step (no tree), same unit;
 *   w[i] >= 0:       weights (NULL: all 1), e.g. decaying with age for an online refit.
 * In units of t_base it fits, by weighted least squares,
 *   lambda * n                      to t_draft / t_base            (beta = 0),
 *   gamma * (exp(delta * n^rho) - 1) to (t_verify - t_base) / t_base (eta = 0),
 * lambda and gamma >= 0 in closed form, (delta, rho) by a refined grid search
 * over rho in [1, 4] and delta * max(n)^rho in [1e-6, 30].
 *   p (or NULL):    lambda, gamma, delta, rho set, beta = eta = 0, other fields untouched;
 *   coef (or NULL): double[4] = lambda, gamma, delta, rho;
 *   rms (or NULL):  double[2] = weighted root-mean-square residual of the draft and of the
 *                   verification fit, in units of t_base.
 * Returns SPEC_TREE_E_PARAM for a null input, npts out of range, a non-finite
 * or negative value, a size <= 0, t_base <= 0 or all weights zero.
 */
int spec_tree_smart_fit(int npts, const double* n, const double* t_draft, const double* t_verify,
                        double t_base, const double* w, spec_tree_params* p, double* coef, double* rms);

/*
 * spec_tree_wait_selftest: a failure-detection check, not a step of the
 * method (the pages have no counterpart).  Every wait inside the library's
 * kernels (on a bulk copy, a ring slot, another warp or another CTA of a
 * cluster) is bounded: after its poll limit it gives up, the kernel ORs
 * SPEC_TREE_S_TIMEOUT into `status`, finishes without waiting again and
 * returns, so that the context stays usable.  This entry point exercises
 * exactly that: one cluster of two CTAs each waits, with `polls` polls (each
 * poll suspends the thread for at most 20 us), on an mbarrier that nothing
 * arrives on, CTA 0 with the CTA-scope wait, CTA 1 with the cluster-scope
 * wait; no copy is in flight.  Each gives up and reports it.
 *   polls:  1 .. 65536 (the kernels' own limit);
 *   status: device uint32, SPEC_TREE_S_TIMEOUT is OR-ed in;
 *   result: device uint32[4]: [2 r] = 1 if CTA r's wait gave up, [2 r + 1] =
 *           the polls it made.
 * Returns SPEC_TREE_E_PARAM for a null pointer or polls out of range.
 */
int spec_tree_wait_selftest(uint32_t polls, uint32_t* status, uint32_t* result, spec_tree_stream_t stream);

/* Message for a return code (static string). */
const char* spec_tree_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_TREE_H */
