/*
 * specverify.h -- C ABI of libspecverify, the GB300 (sm_103a) implementation
 * of the speculative-sampling verification step.
 *
 * The operation (sources cited by page title and section):
 *   [L17] CMU 15-779 Lecture 17 notes, "Speculative Decoding": sec. 2.2
 *         (greedy verification), 2.3 (speculative sampling: accept x ~ q
 *         with probability min(1, p(x)/q(x)), otherwise resample from
 *         norm(max(0, p - q))), 2.4 (Algorithm 1: gamma drafts, one target
 *         pass over gamma+1 positions, stop at the first rejection, bonus
 *         token from p_{gamma+1}), 4.3-4.5 (token trees in depth-first
 *         order, VerifyGreedy, multi-step speculative sampling).
 *   [S14] "Speculative decoding" tutorial (llminference s14): verify(
 *         draft_tokens, q_probs, p_probs, rng) returns the accepted drafts
 *         plus one token; the engine truncates the KV cache by
 *         K - accepted drafts.
 *   [N02] "LLM speculative decoding study notes 02": sec. 3 (r_i ~ U[0,1]),
 *         4 (algorithm), 5.4 (p and q use the same decoding strategy:
 *         temperature, top-k), 10 (greedy), 11.3 (deterministic RNG per
 *         request; drafts of different lengths padded to one K).
 *   [DVP] "Speculative decoding: draft, verify and payoff", II.2 (the
 *         round, KV rollback to the rejected position).
 *
 * Co-residency: the streaming engine's CTAs wait on one another's results
 * (bounded waits), so it is launched cooperatively: every CTA of its grid
 * (one per SM of the device) is resident at once, or the launch fails with
 * SV_ECORESIDENT.  A caller that confines the library to part of the GPU
 * (green contexts, MPS active-thread limits) gets that status rather than
 * timeouts.  The tree walk and the row-statistics kernel wait only inside
 * a thread-block cluster, which the hardware schedules as a unit; the
 * top-k pass waits only within a CTA.
 *
 * Conventions for every entry point:
 *   - All array arguments are DEVICE pointers owned by the caller; the
 *     library allocates nothing and keeps no state between calls except what
 *     lives in the caller's workspace.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  The returned status covers host-side argument
 *     checks and launch errors only; errors found while the kernel reads the
 *     data are recorded in the workspace and read with sv_get_error().
 *   - A workspace must be zeroed once with sv_workspace_init() before its
 *     first use.  Every call leaves each word it wrote zeroed again (the
 *     role that reads a word last clears it), whatever the sizes, so one
 *     workspace (large enough for each call) serves chain and tree calls of
 *     any shape in sequence; after a device error it must be
 *     re-initialised.  One workspace serves one call at a time: calls that
 *     may overlap on the GPU need separate workspaces.
 *   - Status codes are never negative.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* sv_stream_t; /* identical to cudaStream_t */

typedef enum {
  SV_OK = 0,
  SV_EINVAL = 1,      /* bad argument (null pointer, size out of range ...) */
  SV_ECUDA = 2,       /* a CUDA runtime call failed (launch, memcpy ...) */
  SV_ETIMEOUT = 3,    /* a bounded device wait expired (see sv_get_error) */
  SV_EDATA = 4,       /* the data broke a precondition (see sv_get_error) */
  SV_EWORKSPACE = 5,  /* workspace null, too small or misaligned */
  SV_EUNSUPPORTED = 6, /* no sm_103a device / kernel image for this device */
  SV_ECORESIDENT = 7   /* the grid cannot be resident at once (fewer SMs free
                          than the device has: a green context, MPS limits) */
} sv_status;

typedef enum { SV_BF16 = 0, SV_FP32 = 1 } sv_dtype;

typedef enum {
  /* SpecInfer multi-step speculative sampling: child c is tested against
     the draft row q_row[c] as given ([L17] sec. 4.5).  Lossless when the
     children were drawn i.i.d. from their draft rows. */
  SV_TREE_MSS = 0,
  /* MSS for children drawn WITHOUT replacement ([L17] sec. 4.5, the
     precondition of the proof, and sec. 10 exercise 7, the fix): the j-th
     child tried at a node is tested, and the residual formed, against
     q_j = q_row[c] with the tokens of the siblings tried before it removed
     and renormalised; a q_j with no mass left is zero everywhere. */
  SV_TREE_MSS_NOREPLACE = 1,
  /* Naive sampling ([L17] sec. 4.5), the baseline MSS improves on: at the
     current node draw x from p_node by inverse CDF with u_accept[node];
     move to the first child whose token is x, else emit x.  Draft rows are
     not read (draft_logits may be NULL) and u_sample is unused. */
  SV_TREE_NAIVE = 2
} sv_tree_mode;

/* Device error flags, OR-ed into the workspace error word. */
#define SV_DERR_TOKEN 0x01     /* a draft / node token outside [0, V) */
#define SV_DERR_NONFINITE 0x02 /* NaN or +inf in a logit row the step reads */
#define SV_DERR_MASS 0x04      /* a distribution with no mass (all -inf) */
#define SV_DERR_TREE 0x08      /* parent / q_row / depth breaks the format */
#define SV_DERR_TIMEOUT 0x10   /* a bounded wait on a bulk copy expired */
#define SV_DERR_ARG 0x20       /* num_drafts, temperature or top_k invalid */
#define SV_DERR_CHECK 0x40     /* an internal bounds or alignment check failed (debug
                                  builds, -DSV_CHECKS, only): a library bug, never the
                                  data; the access it guarded was skipped */

/* Limits of this implementation. */
#define SV_MAX_K 32        /* drafts per chain */
#define SV_MAX_B 1024      /* requests per call */
#define SV_MAX_V (1 << 20) /* vocabulary entries */
#define SV_MAX_TOPK 64     /* top-k filter size */
#define SV_MAX_TREE_NODES 64 /* nodes per tree (N) and draft rows (M) */
#define SV_MAX_TREE_B 1024  /* requests per tree call */

/*
 * Chain verification, one request per b ([L17] sec. 2.4 Algorithm 1).
 *
 * For request b with nd = num_drafts[b] (or K), temperature t = temperature[b]
 * and top-k k = top_k[b] (0 or >= V: no filter):
 *   p_i = softmax(target row i / t) and q_i = softmax(draft row i / t), both
 *   restricted to their own top-k set (k largest, ties to the lower id);
 *   for i = 0..nd-1: accept x_i iff u_i * q_i(x_i) < p_i(x_i); stop at the
 *   first rejection n and emit one token drawn from norm(max(0, p_n - q_n))
 *   by inverse CDF over ascending token id with u_K; if all nd are accepted,
 *   emit the bonus token drawn from p_nd with u_K.
 *   t == 0 (greedy): accept x_i iff x_i == argmax target row i (lowest id on
 *   ties); emit argmax of target row n.  Draft rows and uniforms are unused.
 *
 * Layout: row i of request b starts at element (b*(K+1) + i) *
 * target_row_stride of target_logits (row_stride >= V), likewise draft rows
 * at (b*K + i) * draft_row_stride.  Rows whose byte address and stride are
 * multiples of 16 (bf16: V a multiple of 8) take the bulk-copy path; others
 * a slower direct path.
 *
 * With a top_k array and max_top_k > 0 the call launches two kernels on the
 * stream: a pass that reduces every filtered row to its top-k (logit, id)
 * list and (max, sum of exp) in the workspace, then the verification kernel,
 * which reads no filtered row itself and finalizes filtered requests from
 * those lists.  Otherwise one kernel.
 */
typedef struct {
  int32_t B, K, V;
  sv_dtype dtype;
  const void* target_logits;   /* [B][K+1][row_stride] */
  int64_t target_row_stride;   /* elements between consecutive rows */
  const void* draft_logits;    /* [B][K][row_stride]; may be NULL when every
                                  request is greedy */
  int64_t draft_row_stride;
  const int32_t* draft_tokens; /* [B][K] */
  const int32_t* num_drafts;   /* [B] in [0, K], or NULL (= K) */
  const float* temperature;    /* [B]; 0 = greedy; < 0 or NaN -> SV_DERR_ARG */
  const int32_t* top_k;        /* [B] or NULL; 0 or >= V = no filter; a
                                  filter keeps the top_k largest logits of p
                                  and of q (ties: lower id first) and must be
                                  <= max_top_k (else SV_DERR_ARG) */
  int32_t max_top_k;           /* host-known bound on top_k (0 = none);
                                  sizes the workspace's top-k lists */
  const float* uniforms;       /* [B][K+1] in [0,1): [0..K-1] accept tests,
                                  [K] the residual / bonus draw */
  int32_t* out_tokens;         /* [B][K+1]: accepted drafts then the emitted
                                  token, -1 padded */
  int32_t* out_len;            /* [B] = accept_len + 1 (0 on a data error) */
  int32_t* accept_len;         /* [B] = accepted drafts = KV truncation
                                  index ([S14] "step": n_rejected = K - it) */
  float* p_at_draft;           /* optional [B][K]: p_i(x_i), NaN unused */
  float* q_at_draft;           /* optional [B][K]: q_i(x_i), NaN unused */
} sv_chain_args;

/*
 * Token-tree verification ([L17] sec. 4.4 VerifyGreedy, 4.5 MSS).
 *
 * Request b holds a tree of n = num_nodes[b] nodes in depth-first order:
 * node 0 is the root (the last verified token; its token is ignored) and
 * 0 <= parent[c] < c for c >= 1.  Target row c is the target distribution
 * after the path root..c; draft row q_row[c] is the draft distribution that
 * proposed node c (siblings may share it).  Starting at the root: children
 * of the current node are tried in ascending index order against the
 * residual r (initially p_node): accept c iff u_accept[c] * q(x_c) < r(x_c)
 * and move to c; on rejection r <- norm(max(0, r - q)).  All rejected: emit
 * a draw from r with u_sample; a node without children: emit a draw from
 * p_node.  Greedy (t == 0): move to the first child whose token is argmax
 * p_node, else emit that argmax.
 *
 * Layout: target row c of request b at (b*N + c) * target_row_stride,
 * draft row m at (b*M + m) * draft_row_stride.
 *
 * Each request is walked by one thread-block cluster that reads only the
 * rows on its path (the target rows of the nodes it stands on, the draft
 * rows its children are tested against, and the next step's rows ahead of
 * time); rows too long for the cluster's shared memory (bf16 V above about
 * 160 K) take a slower engine that reduces every row first.
 */
typedef struct {
  int32_t B, N, M, V, max_depth;
  sv_dtype dtype;
  sv_tree_mode mode;
  const void* target_logits;   /* [B][N][row_stride] */
  int64_t target_row_stride;
  const void* draft_logits;    /* [B][M][row_stride] */
  int64_t draft_row_stride;
  const int32_t* node_tokens;  /* [B][N] */
  const int32_t* parent;       /* [B][N] */
  const int32_t* q_row;        /* [B][N] in [0, M) for c >= 1 */
  const int32_t* num_nodes;    /* [B] in [1, N], or NULL (= N) */
  const float* temperature;    /* [B] */
  const int32_t* top_k;        /* [B] or NULL */
  int32_t max_top_k;
  const float* u_accept;       /* [B][N] */
  const float* u_sample;       /* [B] */
  int32_t* out_tokens;         /* [B][max_depth+1], -1 padded */
  int32_t* out_len;            /* [B] */
  int32_t* accept_len;         /* [B] accepted nodes */
  int32_t* accepted_nodes;     /* [B][max_depth]: node ids along the accepted
                                  path (the KV entries to keep), -1 padded */
} sv_tree_args;

/* Workspace bytes a chain / tree call needs (0 on invalid sizes). */
size_t sv_chain_workspace_bytes(int32_t B, int32_t K, int32_t V, sv_dtype dtype,
                                int32_t max_top_k);
size_t sv_tree_workspace_bytes(int32_t B, int32_t N, int32_t M, int32_t V,
                               sv_dtype dtype, int32_t max_top_k);

/* Zero a workspace (cudaMemsetAsync on `stream`). */
sv_status sv_workspace_init(void* workspace, size_t ws_bytes, sv_stream_t stream);

/* Enqueue one chain / tree verification on `stream`.  The workspace must be
   256-byte aligned and at least the size the matching *_workspace_bytes
   call returns. */
sv_status sv_verify_chain(const sv_chain_args* args, void* workspace,
                          size_t ws_bytes, sv_stream_t stream);
sv_status sv_verify_tree(const sv_tree_args* args, void* workspace,
                         size_t ws_bytes, sv_stream_t stream);

/*
 * Tree-attention mask and depth position ids ([L17] sec. 4.3, tree
 * attention: the tree is laid out depth first; a node attends to the
 * verified prefix, its ancestors and itself; a node's position is its
 * depth; sec. 10 exercise 5).  The step that comes before the tree is
 * verified: the target model's forward pass over the tree uses them.
 *
 * Request b holds n = num_nodes[b] nodes (NULL: N) in depth-first order
 * with parent[b][0] == -1 and 0 <= parent[b][i] < i.  Outputs, row i of
 * request b:
 *   mask[(b*N + i)*words + j/32] bit j%32 is set iff node j is node i or
 *   one of its ancestors (j < N; words beyond the second are zero);
 *   depth[b*N + i] = edges from the root (the position offset after the
 *   verified prefix).
 * Rows i >= n are zero with depth -1.  A malformed tree records
 * SV_DERR_TREE (n outside [1, N]: SV_DERR_ARG) and all its rows are zero
 * with depth -1.  Only the workspace's error word is used: any workspace of
 * at least SV_MIN_WORKSPACE_BYTES (zeroed by sv_workspace_init) will do.
 */
#define SV_MIN_WORKSPACE_BYTES 8192u

typedef struct {
  int32_t B, N;               /* B <= SV_MAX_TREE_B, 1 <= N <= SV_MAX_TREE_NODES */
  int32_t words;              /* 32-bit words per mask row, >= (N + 31) / 32 */
  const int32_t* parent;      /* [B][N] */
  const int32_t* num_nodes;   /* [B] in [1, N], or NULL (= N) */
  uint32_t* mask;             /* [B][N][words] */
  int32_t* depth;             /* [B][N] */
} sv_tree_mask_args;

sv_status sv_tree_mask(const sv_tree_mask_args* args, void* workspace, size_t ws_bytes,
                       sv_stream_t stream);

/*
 * Per-position acceptance statistics of a chain round ([L17] sec. 2.3,
 * Thm 3.5: the draft at position i is accepted with probability
 * alpha_i = sum_x min(p_i(x), q_i(x)) = 1 - TV(p_i, q_i); [N02] sec. 7:
 * E[N] = (1 - a^(K+1)) / (1 - a) when every alpha_i = a).  The inputs an
 * adaptive draft length or an on/off switch for speculation would use.
 *
 * Reads the target, draft, num_drafts, temperature, top_k and max_top_k
 * fields of a chain call's arguments (B, K, V, dtype and strides as there;
 * tokens, uniforms and the outputs are not used and may be NULL).  Outputs:
 *   alpha [B][K]: alpha_i for i < num_drafts[b], NaN beyond.  Greedy
 *     requests (t == 0) have one-hot p and q: alpha_i = 1 iff argmax p_i ==
 *     argmax q_i (lowest id on ties), else 0.  With a top-k filter p_i and
 *     q_i are each restricted to their own top-k set ([N02] sec. 5.4), so
 *     alpha_i sums min(p_i, q_i) over the tokens both sets hold.
 *   expected [B]: sum_{j=0..nd} prod_{i<j} alpha_i, the expected number of
 *     tokens the round emits under these rates.
 * With a top_k array and max_top_k > 0 the call first runs the chain's
 * top-k pass (the same lists sv_verify_chain builds) and needs a workspace
 * of sv_chain_workspace_bytes(B, K, V, dtype, max_top_k) bytes; a filter
 * above max_top_k, or any filter when max_top_k is 0, is reported as
 * SV_DERR_ARG, like a bad num_drafts or temperature.  NaN or +inf logits
 * give SV_DERR_NONFINITE, a row without mass SV_DERR_MASS.  The failing
 * request gets NaN.  Without top-k lists the workspace only needs its
 * header and per-request counters (any sv_chain_workspace_bytes size); what
 * the call uses is left zeroed.
 */
sv_status sv_row_stats(const sv_chain_args* args, float* alpha, float* expected,
                       void* workspace, size_t ws_bytes, sv_stream_t stream);

/* Synchronise `stream`, read and clear the workspace error word.
   *device_flags receives the SV_DERR_* bits (may be NULL).  Returns SV_OK,
   SV_EDATA, SV_ETIMEOUT (when the timeout bit is set) or SV_ECUDA. */
sv_status sv_get_error(void* workspace, sv_stream_t stream, int32_t* device_flags);

/* Self-test of the bounded device wait: one CTA waits on an mbarrier that
   nothing arrives at, with a limit of limit_ns nanoseconds, then reports
   through the workspace error word.  Synchronises `stream`.  Returns
   SV_ETIMEOUT when the wait expired as it must. */
sv_status sv_selftest_wait_timeout(void* workspace, size_t ws_bytes,
                                   int64_t limit_ns, sv_stream_t stream);

/* ---- Allocation-free chain entry point (no counterpart on the pages) ----
 *
 * For callers that cannot hand the library a workspace buffer: a host
 * program with no device allocator of its own at the call site, or a call
 * site where allocating device memory is not allowed or could block.  The
 * scratch these calls use is one file-scope device array per device,
 * SV_NOALLOC_SCRATCH_BYTES long, reserved when the library's module loads;
 * the calls themselves allocate nothing.
 *
 *   - Every call looks up the array's address on the current device
 *     (cudaGetSymbolAddress).  The first call in a context (after a device
 *     reset too) zeroes it on `stream` (cudaMemsetAsync), ahead of the
 *     kernel; make that first call before any stream capture that should
 *     contain only the verification.
 *   - A call whose sv_chain_workspace_bytes(...) exceeds
 *     SV_NOALLOC_SCRATCH_BYTES is rejected with SV_EWORKSPACE before any
 *     device work; use sv_verify_chain with a caller workspace instead.
 *   - The counters at the start of the scratch must be zero when a call
 *     starts; every call leaves them zero.  sv_noalloc_get_error re-zeroes
 *     the scratch (on `stream`) after reporting a device error.
 *   - All calls on one device share the one scratch: calls that may overlap
 *     on the GPU (e.g. on different streams without ordering) race and give
 *     undefined results.  Order them, or use sv_verify_chain with separate
 *     workspaces.
 * Arguments, layouts and results are those of sv_verify_chain. */
#define SV_NOALLOC_SCRATCH_BYTES (8u << 20) /* 8 MiB per device */

sv_status sv_verify_chain_noalloc(const sv_chain_args* args, sv_stream_t stream);

/* sv_get_error for the allocation-free scratch of the current device; after
   a device error it also re-zeroes the scratch on `stream`. */
sv_status sv_noalloc_get_error(sv_stream_t stream, int32_t* device_flags);

const char* sv_status_string(sv_status status);

/* Library version, major*10000 + minor*100 + patch. */
int32_t sv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
