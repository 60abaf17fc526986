/*
 * vt.h - C ABI of libvt: the data-parallel hot path of drafter-based
 * speculative decoding with a VocabTrim-trimmed drafter head, on one GPU.
 *
 * Pages that define the operations (cited by title and section):
 *  [VT]  "VocabTrim: Vocabulary Pruning for Efficient Speculative Decoding in
 *        LLMs" (arXiv 2506.22694): section 3, Algorithm 1 and eq. (1);
 *        Appendix C.1, Algorithm 2.
 *  [GL]  "Speculative decoding" (SelfMadeQuant glossary): sections "Propose a
 *        block, keep a prefix", "Why a rejection needs a special draw",
 *        "Distributional exactness has conditions".
 *  [NB]  "A rejection rule keeps speculative decoding's output exact" (the
 *        nightly build): sections "A target and a draft small enough to print
 *        in full" (the inverse-CDF sampler) and "Extending the rule from one
 *        token to a drafted run" (block verification and the bonus draw).
 *
 * Conventions for every entry point:
 *  - All array pointers are DEVICE pointers owned by the caller; the library
 *    keeps no pointer after the call returns and frees nothing.
 *  - bf16 arrays are passed as uint16_t bit patterns (bfloat16).
 *  - Arrays are dense, row-major, with the strides stated per argument.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *    call is asynchronous on `stream`; the return code reports only what the
 *    host can check (arguments, workspace size, launch errors).
 *  - Problems found in the DATA are reported by the device in *dev_status as
 *    a bit mask of VT_DEV_* flags; the call zeroes *dev_status first.  Read
 *    it after synchronising the stream.  When a VT_DEV_BAD_* or
 *    VT_DEV_NONFINITE bit is set, the affected outputs are unspecified.
 *  - `workspace` is caller-allocated device scratch of at least the size the
 *    matching *_workspace_bytes() query returns, 256-byte aligned.  Its
 *    contents need not be initialised.  Two calls that are in flight at the
 *    same time must not share a workspace.
 *  - Consecutive kernels of the library on one stream overlap through
 *    programmatic dependent launch: a kernel waits for its predecessor
 *    before it touches anything an earlier kernel wrote, with one
 *    exception.  The drafting projection starts streaming W_trim before
 *    that wait, so W_trim must not be written by a kernel that may still be
 *    running when the call's first kernel starts: written by vt_trim_head
 *    (whose last kernel releases no dependent early), by a copy, or by a
 *    kernel of the caller that does not trigger its dependents early.
 *  - The library holds no random number generator: every uniform the method
 *    draws is an explicit input in [0, 1).
 *  - Device code targets sm_103a only.
 */
#ifndef VT_H_
#define VT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
enum {
  VT_OK = 0,
  VT_ERR_INVALID_ARG = -1,  /* null pointer, bad size, bad temperature ...  */
  VT_ERR_UNSUPPORTED = -2,  /* valid request this build does not implement */
  VT_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed         */
  VT_ERR_BAD_INPUT = -4,    /* reserved for host-detected bad data          */
  VT_ERR_WORKSPACE = -5,    /* workspace missing, too small or misaligned  */
  VT_ERR_SCRATCH_LIMIT = -6 /* problem needs more scratch than the library's
                               static array holds (vt_verify_noalloc)      */
};

/* Element types of target logits. */
enum { VT_F32 = 0, VT_BF16 = 1 };

/* Bits the device sets in *dev_status. */
enum {
  VT_DEV_BAD_ID = 1,         /* token id outside [0, V)                        */
  VT_DEV_DUPLICATE_ID = 2,   /* the same id appears twice in a top-K list      */
  VT_DEV_BAD_DRAFT = 4,      /* drafted token out of range, not trimmed, or
                                q(x) <= 0 at a drafted token                    */
  VT_DEV_NONFINITE = 8,      /* NaN/Inf reached a softmax normaliser           */
  VT_DEV_ZERO_RESIDUAL = 16, /* informational: residual mass was zero at a
                                rejection; that draw used p instead            */
  VT_DEV_TIMEOUT = 32        /* a bounded internal wait gave up after about a
                                second (a pipeline mbarrier, or a count another
                                thread block publishes); the affected outputs
                                are unset                                       */
};

/* Human-readable text for a return code. Never NULL. */
const char* vt_status_string(int status);

/* ABI version (major * 100 + minor). */
int vt_abi_version(void);

/* ------------------------------------------------------------------------
 * Calibration: token-frequency histogram and Top-K selection.
 * [VT] Algorithm 1 (a counter c in N^|V| starts at zero and is incremented
 * once per token occurrence) and eq. (1) Top-K(c, k).  Ties in the count are
 * broken by the lower token id.
 *
 *  ids       int32 [n]       calibration token ids, each in [0, V)
 *  n         number of ids (>= 0)
 *  V         vocabulary size (1 <= V <= 2^30; V > 2^22 returns
 *            VT_ERR_UNSUPPORTED in this build)
 *  K         number of ids kept (1 <= K <= V)
 *  counts    uint32 [V]      out: c[t] = occurrences of t (ids outside
 *                            [0, V) are skipped and flag VT_DEV_BAD_ID)
 *  topk_ids  int32 [K]       out: the K ids ranked by (count desc, id asc)
 *  dev_status int32 [1]      out: VT_DEV_* bits
 * Counts are exact (bit-identical to a sequential count) for n < 2^32.
 * Workspace: vt_calibrate_topk_workspace_bytes(n, V, K) bytes, about
 * 28 bytes per id of V (0 when V > 2^22).
 * ---------------------------------------------------------------------- */
size_t vt_calibrate_topk_workspace_bytes(int64_t n, int32_t V, int32_t K);
int vt_calibrate_topk(const int32_t* ids, int64_t n, int32_t V, int32_t K,
                      uint32_t* counts, int32_t* topk_ids, int32_t* dev_status,
                      void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Vocabulary selection by Top-P or by a minimum frequency.  [VT] section 3
 * notes that the trimmed vocabulary may also be chosen by Top-P or by the
 * minimum frequency of tokens in the calibration data instead of Top-K; the
 * page defines neither, and these entry points take the plainest readings:
 *  vt_calibrate_top_p      K = the smallest prefix length of the ranking
 *                          whose counts reach P * (sum of all counts),
 *                          compared in fp64; 0 < P <= 1; K = 0 when no id
 *                          was counted
 *  vt_calibrate_min_count  K = the number of ids counted at least min_count
 *                          times (they are the first K of the ranking)
 *
 *  ids, n, V      as vt_calibrate_topk (V <= 2^22)
 *  counts     uint32 [V]   out: c[t]
 *  ranked_ids int32  [V]   out: all V ids ranked (count desc, id asc)
 *  k_out      int32  [1]   out, device memory: K.  Read it once the stream
 *                          has synchronised; ranked_ids[0..K) is the
 *                          selection, ready for vt_trim_head.
 *  dev_status int32  [1]   out: VT_DEV_BAD_ID, VT_DEV_TIMEOUT
 * Workspace: vt_calibrate_select_workspace_bytes(n, V) bytes (0 when V is
 * out of range).  P outside (0, 1] or non-finite: VT_ERR_INVALID_ARG.
 * ---------------------------------------------------------------------- */
size_t vt_calibrate_select_workspace_bytes(int64_t n, int32_t V);
int vt_calibrate_top_p(const int32_t* ids, int64_t n, int32_t V, double P,
                       uint32_t* counts, int32_t* ranked_ids, int32_t* k_out,
                       int32_t* dev_status, void* workspace, size_t workspace_bytes,
                       void* stream);
int vt_calibrate_min_count(const int32_t* ids, int64_t n, int32_t V, uint32_t min_count,
                           uint32_t* counts, int32_t* ranked_ids, int32_t* k_out,
                           int32_t* dev_status, void* workspace, size_t workspace_bytes,
                           void* stream);

/* ------------------------------------------------------------------------
 * Trimmed LM head.  [VT] eq. (1): W^Trim = W[Top-K(c,k), :]; Algorithm 2's
 * token index mapper T_{d->t} (trimmed index -> target id) and its inverse.
 * Rows are kept in ascending target-id order.
 *
 *  W         bf16 [V, H]     full LM head, row stride H
 *  topk_ids  int32 [K]       K distinct ids in [0, V), any order
 *  W_trim    bf16 [K, H]     out: W_trim[j, :] = W[trim_ids[j], :] bit for bit
 *  trim_ids  int32 [K]       out: the selected ids, ascending (T_{d->t})
 *  inv_map   int32 [V]       out: inv_map[trim_ids[j]] = j, -1 elsewhere
 *  dev_status int32 [1]      out: VT_DEV_BAD_ID / VT_DEV_DUPLICATE_ID
 * Workspace: vt_trim_head_workspace_bytes(V, K) bytes (8 bytes per 32 ids).
 * ---------------------------------------------------------------------- */
size_t vt_trim_head_workspace_bytes(int32_t V, int32_t K);
int vt_trim_head(const uint16_t* W, int32_t V, int32_t H,
                 const int32_t* topk_ids, int32_t K,
                 uint16_t* W_trim, int32_t* trim_ids, int32_t* inv_map,
                 int32_t* dev_status, void* workspace, size_t workspace_bytes,
                 void* stream);

/* ------------------------------------------------------------------------
 * Drafter logits through the trimmed head.  [VT] Algorithm 2, drafting
 * (the trimmed drafter scores only the K trimmed ids); temperature divides
 * the logits ([GL] "Distributional exactness has conditions").
 *
 *  hidden    bf16 [B, H]     drafter hidden states, row stride H
 *  W_trim    bf16 [K, H]     trimmed head
 *  logits    f32  [B, ld_logits] out: logits[b, j] = (sum_h hidden[b,h] *
 *            W_trim[j,h]) / T, accumulated in fp32; ld_logits >= K
 * 1 <= B <= 4096, 1 <= H <= 65536, 1 <= K; T finite and > 0.
 * ---------------------------------------------------------------------- */
size_t vt_draft_workspace_bytes(int32_t B, int32_t H, int32_t K);
int vt_draft_logits(const uint16_t* hidden, int32_t B, int32_t H,
                    const uint16_t* W_trim, int32_t K, float temperature,
                    float* logits, int64_t ld_logits,
                    void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * One drafting step.  [VT] Algorithm 2, drafting: logits over the trimmed
 * vocabulary, q = softmax(logits / T), one categorical draw per row, mapped
 * to a target id by trim_ids.  The draw is the inverse CDF of [NB] with a
 * strict comparison: the smallest trimmed index j whose running sum of q
 * (ascending j, i.e. ascending target id) exceeds u_b * sum(q); if rounding
 * leaves none, the last j with q_j > 0.
 *
 *  hidden    bf16 [B, H]     drafter hidden states
 *  W_trim    bf16 [K, H]     trimmed head
 *  trim_ids  int32 [K]       trimmed index -> target id
 *  uniforms  f32  [B]        one uniform in [0,1) per row
 *  q         f32  [B, ldq]   out: q[b, j] for j < K (ldq >= K; pass
 *                            ldq = gamma*K and q + pos*K to fill position
 *                            `pos` of a [B, gamma, K] tensor)
 *  tokens    int32 [B, ld_tokens] out: drafted target ids in column 0
 *                            (pass ld_tokens = gamma and tokens + pos to fill
 *                            column `pos` of a [B, gamma] tensor; ld_tokens >= 1)
 *  dev_status int32 [1]      out: VT_DEV_NONFINITE
 * T == 0 drafts greedily ([VT] section 4 decodes greedily; Algorithm 2):
 * j* = the largest logit of row b, ties to the lower trimmed index (the
 * lower target id), q[b, :] = one-hot at j* (the limit of softmax(z/T)),
 * token = trim_ids[j*]; uniforms are not read and may be NULL.  T < 0 or
 * non-finite: VT_ERR_INVALID_ARG.
 * ---------------------------------------------------------------------- */
int vt_draft_step(const uint16_t* hidden, int32_t B, int32_t H,
                  const uint16_t* W_trim, const int32_t* trim_ids, int32_t K,
                  const float* uniforms, float temperature,
                  float* q, int64_t ldq, int32_t* tokens, int64_t ld_tokens,
                  int32_t* dev_status, void* workspace, size_t workspace_bytes,
                  void* stream);

/* ------------------------------------------------------------------------
 * The drafter's top-k candidates at one position: the expansion step of a
 * draft tree ([VT] section 4.1 grows EAGLE-2 trees with top-K 8 through the
 * trimmed head).  z as in vt_draft_logits; the k highest z of row b, ties
 * to the lower trimmed index, best first, mapped to target ids, each with
 * log q = log softmax(z / T) over the trimmed vocabulary.  How a tree is
 * grown from them (which nodes to expand, re-ranking) is the caller's.
 *
 *  out_ids  int32 [B, k]  out: target ids (-1 for a row with non-finite z)
 *  out_logq f32   [B, k]  out: log q of each (NaN for such a row)
 *  dev_status int32 [1]   out: VT_DEV_NONFINITE
 * 1 <= k <= 32 and k <= K (else VT_ERR_INVALID_ARG); T finite and > 0.
 * Workspace:
 * vt_draft_topk_workspace_bytes(B, H, K, k) bytes.
 * ---------------------------------------------------------------------- */
size_t vt_draft_topk_workspace_bytes(int32_t B, int32_t H, int32_t K, int32_t k);
int vt_draft_topk(const uint16_t* hidden, int32_t B, int32_t H, const uint16_t* W_trim,
                  const int32_t* trim_ids, int32_t K, int32_t k, float temperature,
                  int32_t* out_ids, float* out_logq, int32_t* dev_status,
                  void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Batched block verification by modified rejection sampling.
 * [GL] "Why a rejection needs a special draw": accept a drafted x with
 * probability a(x) = min(1, p(x)/q(x)); on rejection draw from
 * norm(max(p - q, 0)) over the full vocabulary.  [GL] "Propose a block, keep
 * a prefix" and [NB] "Extending the rule ...": test left to right, keep the
 * accepted prefix, replace the first rejected token with the residual draw
 * made from THAT position's p and q, discard the rest; if all gamma drafts
 * are accepted, draw a bonus token from p at position gamma.
 * p_i = softmax(logits[b, i, :] / T) over all V ids; q_i is zero outside the
 * trimmed vocabulary.  Accept iff u_accept[b,i] < a(x).  Every draw is the
 * strict inverse CDF in ascending token-id order (see vt_draft_step).
 *
 *  target_logits  [B, gamma+1, V] of logits_dtype (VT_F32 or VT_BF16)
 *  q         f32  [B, gamma, K]   drafter probabilities over trimmed ids
 *  inv_map   int32 [V]            target id -> trimmed index, -1 if absent
 *  draft_tokens int32 [B, gamma]  drafted target ids
 *  u_accept  f32  [B, gamma]      accept uniforms
 *  u_resample f32 [B, gamma+1]    uniform of the residual (or bonus) draw;
 *                                 entry n_b is used
 *  temperature                    T > 0, the T that produced q; T == 0
 *                                 verifies greedily (below)
 *  out_tokens int32 [B, gamma+1]  out: draft[0..n_b-1], then the drawn
 *                                 token, then -1
 *  out_num_accepted int32 [B]     out: n_b in [0, gamma]
 *  out_accept_prob f32 [B, gamma] out, may be NULL: a(x) at each tested
 *                                 position (0..min(n_b, gamma-1)); NaN at
 *                                 positions after the first rejection
 *  dev_status int32 [1]           out: VT_DEV_BAD_DRAFT, VT_DEV_NONFINITE,
 *                                 VT_DEV_ZERO_RESIDUAL, VT_DEV_TIMEOUT
 * 1 <= gamma <= 64, 1 <= B, 1 <= K <= V <= 2^22.
 *
 * T == 0, greedy verification ([VT] section 4: a drafted token is accepted
 * only if it exactly matches the target's choice; Algorithm 2): position i
 * keeps x_i iff x_i is the largest logit of logits[b, i, :] (ties to the
 * lower id, compared exactly as given); the first mismatch n is replaced by
 * that row's choice and the block ends; with no mismatch the choice at
 * position gamma is appended.  q, inv_map, u_accept and u_resample are not
 * read (may be NULL; K only sizes the workspace).  out_accept_prob is 1 at
 * accepted positions, 0 at the rejected one, NaN after.  dev_status:
 * VT_DEV_BAD_DRAFT (a drafted id outside [0, V) reached by the walk),
 * VT_DEV_NONFINITE.
 * ---------------------------------------------------------------------- */
size_t vt_verify_workspace_bytes(int32_t B, int32_t gamma, int32_t V, int32_t K);
int vt_verify(const void* target_logits, int32_t logits_dtype,
              int32_t B, int32_t gamma, int32_t V,
              const float* q, const int32_t* inv_map, int32_t K,
              const int32_t* draft_tokens, const float* u_accept,
              const float* u_resample, float temperature,
              int32_t* out_tokens, int32_t* out_num_accepted,
              float* out_accept_prob, int32_t* dev_status,
              void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * vt_verify_noalloc - vt_verify for callers that cannot allocate device
 * memory.  The pages have no counterpart of this entry point: it changes
 * nothing in what is computed, only where the scratch lives.
 *
 * Some callers have no way to hand the library a workspace: an extension
 * loaded into a host runtime that owns all device memory and gives its
 * plug-ins no allocator, C code without a device allocator of its own, or a
 * latency-critical loop that must not call cudaMalloc (which can
 * synchronise the whole device).  This variant takes exactly the inputs and
 * outputs of vt_verify, minus the workspace.  Its scratch is a file-scope
 * static device array of VT_VERIFY_NOALLOC_SCRATCH_BYTES (2 MiB) inside
 * libvt, which every GPU that loads the library holds until the process
 * exits.
 *  - Limit: a problem whose vt_verify_workspace_bytes(B, gamma, V, K) is
 *    larger than VT_VERIFY_NOALLOC_SCRATCH_BYTES is rejected with
 *    VT_ERR_SCRATCH_LIMIT before any device work (about 3800 rows
 *    B*(gamma+1) fit, e.g. B=256 with gamma=8).
 *  - Set-up: every call looks up the array's device address
 *    (cudaGetSymbolAddress) in the calling thread's current context and
 *    returns VT_ERR_CUDA if the lookup fails.  Each context that loads the
 *    library has its own copy of the array, so no address is cached: a
 *    call after cudaDeviceReset, or from a context the caller created and
 *    made current itself, uses that context's copy.  The first call in a
 *    context also loads the library's device code there; make it before
 *    any stream capture.
 *  - Arguments are checked exactly as vt_verify checks them (same codes);
 *    the scratch limit is checked after that.
 *  - Sharing: every call on a device uses the same array, which keeps what
 *    the last call left in it; the kernels clear what must start at zero.
 *    Calls that can overlap on the GPU (e.g. on two streams with no ordering
 *    between them) race on the array and give undefined results: order them.
 *  - The call performs no cudaMalloc, cudaFree or other allocation.
 * ---------------------------------------------------------------------- */
#define VT_VERIFY_NOALLOC_SCRATCH_BYTES ((size_t)2 << 20)
int vt_verify_noalloc(const void* target_logits, int32_t logits_dtype,
                      int32_t B, int32_t gamma, int32_t V,
                      const float* q, const int32_t* inv_map, int32_t K,
                      const int32_t* draft_tokens, const float* u_accept,
                      const float* u_resample, float temperature,
                      int32_t* out_tokens, int32_t* out_num_accepted,
                      float* out_accept_prob, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * Greedy verification of draft trees.  [VT] section 4.1 drafts, builds and
 * verifies trees as EAGLE-2 does (depth 3, top-K 8, at most 32 tokens) with
 * the greedy target of section 4; Algorithm 2 keeps the consistent prefix
 * and replaces the first inconsistent token.  A tree holds N drafted nodes
 * in topological order: node i carries tokens[b, i] (a target id) and
 * parent[b, i] in {-1} or [0, i), -1 meaning the context.  The target has
 * scored N + 1 positions: row 0 after the context, row i + 1 after node i
 * (with the tree attention of the caller's target model).
 * Node i is accepted iff its parent is (the context always is) and its
 * token is the largest logit of its parent's row (ties to the lower id,
 * compared exactly as given).  The block is the token path from the context
 * to the deepest accepted node (ties to the lower node index) followed by
 * the target's choice at that node's row; a chain (parent[i] = i - 1) gives
 * exactly vt_verify's greedy block.
 *
 *  target_logits [B, N+1, V] of logits_dtype
 *  parent    int32 [B, N]   (row stride parent_stride >= N, or 0: one tree
 *                            shared by all sequences)
 *  tokens    int32 [B, N]   drafted target ids
 *  temperature              0 (greedy); T > 0 returns VT_ERR_UNSUPPORTED
 *  out_tokens int32 [B, N+1] out: the path's tokens, the target's choice,
 *                            then -1
 *  out_num_accepted int32 [B] out: the path length (accepted tokens)
 *  out_path  int32 [B, N]   out, may be NULL: the path's node indices, -1 after
 *  dev_status int32 [1]     out: VT_DEV_BAD_DRAFT (a token outside [0, V) or
 *                            a parent not before its node; that sequence
 *                            gets -1 tokens), VT_DEV_NONFINITE
 * 1 <= N <= 255, 1 <= B, V <= 2^22.  Workspace:
 * vt_verify_tree_workspace_bytes(B, N, V) bytes.
 * ---------------------------------------------------------------------- */
size_t vt_verify_tree_workspace_bytes(int32_t B, int32_t N, int32_t V);
int vt_verify_tree(const void* target_logits, int32_t logits_dtype, int32_t B, int32_t N,
                   int32_t V, const int32_t* parent, int64_t parent_stride,
                   const int32_t* tokens, float temperature, int32_t* out_tokens,
                   int32_t* out_num_accepted, int32_t* out_path, int32_t* dev_status,
                   void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * One speculative block as a CUDA graph.  [VT] Appendix C.1, Algorithm 2:
 * draft k (= gamma) tokens through the trimmed head, then score and verify
 * them.  vt_block_graph_create records gamma vt_draft_step calls (step j
 * reads hidden[j] and u_draft[j] and writes q[:, j, :] and
 * draft_tokens[:, j]) followed by one vt_verify call, with the
 * programmatic-dependent-launch edges between consecutive kernels, into a
 * CUDA graph on a private stream; vt_block_graph_launch replays the whole
 * block with one launch on `stream`.  A replay computes exactly what the
 * same calls made directly would.
 *
 * The pointers in the descriptor are fixed at creation: a replay reads
 * whatever the input buffers hold when it runs and overwrites the outputs.
 * Layouts (row-major, device memory owned by the caller):
 *  hidden        bf16 [gamma, B, H]      u_draft  f32 [gamma, B] (NULL if T == 0)
 *  W_trim        bf16 [K, H]             trim_ids int32 [K], inv_map int32 [V]
 *  target_logits [B, gamma+1, V] of logits_dtype
 *  u_accept      f32 [B, gamma], u_resample f32 [B, gamma+1] (NULL if T == 0)
 *  q             f32 [B, gamma, K] out   draft_tokens int32 [B, gamma] out
 *  out_tokens    int32 [B, gamma+1] out, out_num_accepted int32 [B] out,
 *  out_accept_prob f32 [B, gamma] out or NULL
 *  dev_status    int32 [2] out: [0] the drafting flags of all gamma steps
 *                (OR), [1] the verification flags
 *  workspace     vt_block_workspace_bytes(B, H, K, V, gamma) bytes, 256-byte
 *                aligned, used by every replay (replays on streams without
 *                an order between them race on it)
 * The sizes follow vt_draft_step and vt_verify; argument errors of those
 * calls are returned by vt_block_graph_create (nothing is created then).
 * *graph receives an opaque handle; vt_block_graph_destroy releases it.
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t B, H, K, V, gamma;
  int32_t logits_dtype;           /* VT_F32 or VT_BF16 */
  float temperature;              /* T > 0, or 0 for the greedy block */
  const uint16_t* hidden;
  const uint16_t* W_trim;
  const int32_t* trim_ids;
  const int32_t* inv_map;
  const float* u_draft;
  const void* target_logits;
  const float* u_accept;
  const float* u_resample;
  float* q;
  int32_t* draft_tokens;
  int32_t* out_tokens;
  int32_t* out_num_accepted;
  float* out_accept_prob;
  int32_t* dev_status;
  void* workspace;
  size_t workspace_bytes;
} vt_block_desc;

size_t vt_block_workspace_bytes(int32_t B, int32_t H, int32_t K, int32_t V, int32_t gamma);
int vt_block_graph_create(const vt_block_desc* desc, void** graph);
int vt_block_graph_launch(void* graph, void* stream);
int vt_block_graph_destroy(void* graph);

/* ---------------------------------------------------------------------------
 * vt_selftest_wait — failure detection self-test of the bounded waits.
 *
 * Not part of the method: it runs, in one thread of one thread block, the
 * same device wait helpers the kernels above use between thread blocks,
 * with a caller-chosen iteration limit, so a test can make a wait give up
 * without anything hanging, and check that the status word says so.
 *   which 0: wait on an mbarrier that nothing arrives on (the wait helper
 *            of the tcgen05 pipelines) -- always gives up;
 *   which 1: the same mbarrier after one arrival -- completes;
 *   which 2: poll *flag until bit 31 is set (the helper with which a radix
 *            sort tile waits for the digit counts of earlier tiles) -- gives
 *            up unless bit 31 of *flag is set.
 * limit    polls before giving up, 1 <= limit <= 2^20.
 * flag     uint32 [1] device, read only (which 2; may be NULL otherwise).
 * dev_status int32 [1] device: VT_DEV_TIMEOUT is OR-ed in when the wait
 *          gives up; nothing else is written.
 * Returns VT_ERR_INVALID_ARG for another `which`, a limit out of range, or a
 * missing pointer; VT_ERR_CUDA if the launch fails.  Asynchronous on `stream`.
 */
int vt_selftest_wait(int32_t which, uint32_t limit, const uint32_t* flag, int32_t* dev_status,
                     void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VT_H_ */
