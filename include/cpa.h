/*
 * cpa.h -- C ABI of the cascade paged-attention library (libcpa.so) for
 * GB300 (sm_103a).
 *
 * The method.  For one query q and a key set split into disjoint parts A and
 * B, attention over A and over B can be computed separately and merged
 * exactly by their log-sum-exp values ("Cascade attention" page,
 * zdszero.github.io/cascade_attention.html, section on the split property):
 *     LSE = log(e^LSE_A + e^LSE_B),  o = e^(LSE_A-LSE) o_A + e^(LSE_B-LSE) o_B.
 * In tree speculative-decoding verify, request b holds a prefix of L_b cached
 * tokens and topk branches of S draft tokens each; draft s of branch k
 * attends the whole prefix plus drafts 0..s of its own branch (same page,
 * "Topk > 1").  Cascade reads the shared prefix once per request (Pass A, all
 * topk*S draft queries of the request together), each branch's own drafts
 * once (Pass B) and merges the two.  Naive expand instead runs B*topk
 * independent requests over L_b + S keys each and so reads every prefix topk
 * times (same page, "Naive Expand").  The same split covers prefill after a
 * prefix-cache hit of H tokens: the M = N - H suffix queries attend the
 * cached prefix (an M x H rectangle) and each other causally (a triangle),
 * merged the same way ("Causal Attention ... KV hit area" page, sections 2-3).
 *
 * Conventions shared by every call.
 *   - Data types: q, k_pages, v_pages and bf16 outputs are bfloat16 (2 bytes);
 *     lse and fp32 outputs are float.  head_dim must be 128.
 *   - Paged KV pool (KV-cache tutorial, sections 5.2-5.3): k_pages and
 *     v_pages are [num_pages, page_size, H_kv, head_dim], row-major.  Logical
 *     position pos of a sequence with block table `tab` is page
 *     tab[pos / page_size], slot pos % page_size.  Slots past a sequence's
 *     end are never used: their contents may be anything, NaN included.
 *   - Grouped-query attention: query head h reads KV head h / (H_q / H_kv)
 *     (repeat_interleave grouping, tutorial section 6.3).  H_q / H_kv must be
 *     a power of two no larger than 128.
 *   - Verify token order: q and o are [B*topk*S, H_q, head_dim] and lse is
 *     [B*topk*S, H_q]; token t = (b*topk + k)*S + s is draft s of branch k of
 *     request b.
 *   - lse is the natural-log log-sum-exp of the scaled scores over the keys a
 *     row sees; a row that sees no key gets lse = -inf and o = 0.
 *   - Pointers passed as `const void*` / `void*` / `float*` / `int32_t*` are
 *     DEVICE pointers (16-byte aligned for q, k_pages, v_pages, o) unless a
 *     comment says host.  The caller owns every buffer, including the
 *     workspace; the library never allocates, frees or synchronises (except
 *     cpa_get_device_status and cpa_noalloc_device_status, which say so).
 *     Calls are asynchronous on `stream` (NULL = legacy default stream) and
 *     launch nothing when they return an error, with one exception:
 *     cpa_cascade_verify_shared launches two kernels when its shared prefix
 *     ends inside a page, and checks every argument before the first, so only
 *     CPA_ERR_LAUNCH or CPA_ERR_CUDA from the second launch can follow a
 *     launch already made.
 *   - Errors: arguments that can be checked on the host return a status
 *     before any launch.  Problems only the GPU can see (a page id outside
 *     [0, num_pages), a prefix length outside [0, max_prefix_len], a pipeline
 *     wait that exceeded its time limit) set bits in a status word at the
 *     start of the workspace, which cpa_get_device_status reads.  Each
 *     workspace-taking call clears that word and the merge counters it uses
 *     (an asynchronous memset on `stream`).  Nothing crosses the ABI as an
 *     exception, and no kernel traps, asserts or prints.
 *   - When the device status word has any bit set after a call, that call's
 *     outputs are undefined (they may be partial, stale or computed from a
 *     truncated mask); only the status word is meaningful.
 *   - A workspace must not be used by two calls that can run at the same time.
 */
#ifndef CPA_H_
#define CPA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* A CUDA stream (cudaStream_t / CUstream). */
typedef struct CUstream_st* cpa_stream_t;

typedef enum cpa_status {
    CPA_OK = 0,
    CPA_ERR_INVALID_ARG = 1,  /* bad pointer, size, stride or shape */
    CPA_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels implement */
    CPA_ERR_WORKSPACE = 3,    /* workspace missing or too small */
    CPA_ERR_LAUNCH = 4,       /* a kernel launch failed */
    CPA_ERR_BAD_PAGE = 5,     /* device saw a page id outside [0, num_pages) */
    CPA_ERR_TIMEOUT = 6,      /* device pipeline wait exceeded its limit */
    CPA_ERR_CUDA = 7,         /* a CUDA runtime call failed */
    CPA_ERR_BAD_LENGTH = 8,   /* device saw a prefix length outside [0, max_prefix_len] */
    CPA_ERR_BAD_TREE = 9      /* device saw a tree parent index outside [-1, i) */
} cpa_status;

/* Bits of the device status word (first 4 bytes of a workspace). */
#define CPA_DEV_BAD_PAGE 0x1u
#define CPA_DEV_TIMEOUT 0x2u
#define CPA_DEV_BAD_LENGTH 0x4u
#define CPA_DEV_BAD_TREE 0x8u

/* Largest draft tree cpa_tree_verify accepts (one 64-bit ancestor mask per node). */
#define CPA_MAX_TREE_NODES 64

/* Which part of the prefix-hit prefill to compute (cpa_prefill_hit). */
#define CPA_PREFILL_FULL 0 /* rectangle + triangle, merged; o is bf16 */
#define CPA_PREFILL_RECT 1 /* keys 0..H-1 only; o is fp32 */
#define CPA_PREFILL_TRI 2  /* keys H..H+i only; o is fp32 */

/* Human-readable name of a status code (static string). */
const char* cpa_status_string(cpa_status status);

/*
 * Bytes of workspace cpa_cascade_verify, cpa_cascade_pass_a and
 * cpa_naive_expand_verify need for these sizes on the current device.  The
 * workspace holds the device status word, one merge counter per work unit
 * and the fp32 partial results of work units that are split across CTAs.
 * Returns 0 for sizes the calls would reject.
 */
size_t cpa_cascade_verify_workspace_size(int B, int topk, int S, int H_q, int H_kv, int head_dim,
                                         int page_size);

/*
 * Cascade verify attention (the whole hot path): Pass A + Pass B + merge.
 *   q                  bf16 [B*topk*S, H_q, head_dim]
 *   k_pages, v_pages   bf16 [num_pages, page_size, H_kv, head_dim]
 *   prefix_page_table  int32 [B, prefix_pt_stride]: request b's prefix pages
 *                      ("metadata.page_table" of the cascade page); entries
 *                      past ceil(L_b / page_size) are not read.
 *   draft_page_table   int32 [B*topk, draft_pt_stride]: branch (b, k)'s draft
 *                      pages ("forward_metadata_spec_decode_expand.page_table");
 *                      draft j is at logical position j of its branch.
 *   prefix_lens        int32 [B] on the device: L_b >= 0 ("cache_seqlens").
 *   max_prefix_len     host-side upper bound of every L_b; prefix_pt_stride
 *                      must be >= ceil(max_prefix_len / page_size).
 *   sm_scale           softmax scale (> 0), normally 1/sqrt(head_dim).
 *   o                  bf16 [B*topk*S, H_q, head_dim] output.
 *   lse                fp32 [B*topk*S, H_q] output (natural log).
 * Supported: head_dim 128; page_size in {8,16,32,64,128,256}; 1 <= S <= 16
 * and S <= page_size (a branch's drafts share its first draft page);
 * topk <= 16 when S <= 8, topk <= 8 when S > 8 (the branches' draft blocks of
 * 8 or 16 rows fill one 128-key tile); topk*S*(H_q/H_kv) <= 256.
 */
cpa_status cpa_cascade_verify(const void* q, const void* k_pages, const void* v_pages,
                              const int32_t* prefix_page_table, int prefix_pt_stride,
                              const int32_t* draft_page_table, int draft_pt_stride,
                              const int32_t* prefix_lens, int B, int topk, int S, int H_q,
                              int H_kv, int head_dim, int page_size, int num_pages,
                              int max_prefix_len, float sm_scale, void* o, float* lse,
                              void* workspace, size_t workspace_bytes, cpa_stream_t stream);

/*
 * Naive-expand verify: the comparison baseline.  Same arguments and result
 * as cpa_cascade_verify, but every branch (b, k) is run as its own request
 * over its L_b + S logical keys (prefix pages, then its own draft pages), so
 * each prefix is read topk times: B*topk*(L+S) KV tokens in total (cascade
 * page, "Naive Expand").  Supported: S*(H_q/H_kv) <= 256, S <= 16,
 * S <= page_size.  Workspace: cpa_cascade_verify_workspace_size.
 */
cpa_status cpa_naive_expand_verify(const void* q, const void* k_pages, const void* v_pages,
                                   const int32_t* prefix_page_table, int prefix_pt_stride,
                                   const int32_t* draft_page_table, int draft_pt_stride,
                                   const int32_t* prefix_lens, int B, int topk, int S, int H_q,
                                   int H_kv, int head_dim, int page_size, int num_pages,
                                   int max_prefix_len, float sm_scale, void* o, float* lse,
                                   void* workspace, size_t workspace_bytes, cpa_stream_t stream);

/*
 * Pass A alone (cascade page, first segment): every draft query of request b
 * against the request's prefix keys 0..L_b-1, read once per request.
 *   o_a   fp32 [B*topk*S, H_q, head_dim];  lse_a fp32 [B*topk*S, H_q].
 * A request with L_b = 0 gives o_a = 0, lse_a = -inf.
 */
cpa_status cpa_cascade_pass_a(const void* q, const void* k_pages, const void* v_pages,
                              const int32_t* prefix_page_table, int prefix_pt_stride,
                              const int32_t* prefix_lens, int B, int topk, int S, int H_q,
                              int H_kv, int head_dim, int page_size, int num_pages,
                              int max_prefix_len, float sm_scale, float* o_a, float* lse_a,
                              void* workspace, size_t workspace_bytes, cpa_stream_t stream);

/*
 * Pass B alone (cascade page, second segment): B*topk virtual requests; draft
 * s of branch (b, k) against that branch's drafts 0..s, one warp per
 * (branch, query head) with a warp-level online softmax.
 *   o_b   fp32 [B*topk*S, H_q, head_dim];  lse_b fp32 [B*topk*S, H_q].
 * The workspace only needs to hold the status word: at least
 * cpa_status_workspace_size() bytes.  Supported: head_dim 128.
 */
cpa_status cpa_cascade_pass_b(const void* q, const void* k_pages, const void* v_pages,
                              const int32_t* draft_page_table, int draft_pt_stride, int B,
                              int topk, int S, int H_q, int H_kv, int head_dim, int page_size,
                              int num_pages, float sm_scale, float* o_b, float* lse_b,
                              void* workspace, size_t workspace_bytes, cpa_stream_t stream);

/* Bytes of workspace that hold only the device status word. */
size_t cpa_status_workspace_size(void);

/*
 * merge_state (cascade page): for each of n_tokens*H rows,
 *   lse = log(e^lse_a + e^lse_b),  o = e^(lse_a-lse) o_a + e^(lse_b-lse) o_b,
 * computed about max(lse_a, lse_b) so nothing overflows; a -inf side
 * contributes nothing and two -inf sides give o = 0, lse = -inf.
 *   o_a, o_b  fp32 [n_tokens, H, head_dim];  lse_a, lse_b fp32 [n_tokens, H]
 *   o_out     bf16 [n_tokens, H, head_dim];  lse_out fp32 [n_tokens, H]
 * Supported: head_dim a multiple of 4 and at most 512.
 */
cpa_status cpa_merge_state(const float* o_a, const float* lse_a, const float* o_b,
                           const float* lse_b, int n_tokens, int H, int head_dim, void* o_out,
                           float* lse_out, cpa_stream_t stream);

/*
 * Cascade verify over FP8 KV pages (KV-cache tutorial, section 4.5 "FP8 KV":
 * half the bytes of bf16, with a per-tensor or per-channel scale).  Same
 * arguments, layout, token order and results as cpa_cascade_verify, except:
 *   k_pages, v_pages   uint8 [num_pages, page_size, H_kv, head_dim] E4M3 codes
 *                      (1 sign, 4 exponent bits with bias 7, 3 mantissa bits;
 *                      exponent 0 holds zero and subnormals); element value =
 *                      decoded code x scale.
 *   k_scale, v_scale   fp32 on the device: one value each when
 *                      scale_per_channel is 0, else [H_kv, head_dim] each
 *                      (one scale per KV head and channel).
 * q stays bf16 and o bf16, lse fp32.  The two NaN codes (0x7F, 0xFF) must not
 * appear in slots a row sees: they are read as +-480 x scale, not as NaN
 * (every other code is exact).  Slots past a sequence's end may hold any byte.
 * Arithmetic: codes are widened exactly to f16 on chip; q x k_scale is
 * rounded to f16 once (so |q x k_scale| must stay below 65504), P is f16,
 * accumulation fp32.  Supported: as for cpa_cascade_verify, and
 * topk*S*(H_q/H_kv) <= 128 (one M tile).  Workspace:
 * cpa_cascade_verify_workspace_size.
 */
cpa_status cpa_cascade_verify_fp8(const void* q, const void* k_pages, const void* v_pages,
                                  const float* k_scale, const float* v_scale,
                                  int scale_per_channel, const int32_t* prefix_page_table,
                                  int prefix_pt_stride, const int32_t* draft_page_table,
                                  int draft_pt_stride, const int32_t* prefix_lens, int B, int topk,
                                  int S, int H_q, int H_kv, int head_dim, int page_size,
                                  int num_pages, int max_prefix_len, float sm_scale, void* o,
                                  float* lse, void* workspace, size_t workspace_bytes,
                                  cpa_stream_t stream);

/*
 * Pass A alone over FP8 KV pages: cpa_cascade_pass_a's result (fp32 o_a,
 * lse_a) with the pools and scales of cpa_cascade_verify_fp8.
 */
cpa_status cpa_cascade_pass_a_fp8(const void* q, const void* k_pages, const void* v_pages,
                                  const float* k_scale, const float* v_scale,
                                  int scale_per_channel, const int32_t* prefix_page_table,
                                  int prefix_pt_stride, const int32_t* prefix_lens, int B,
                                  int topk, int S, int H_q, int H_kv, int head_dim, int page_size,
                                  int num_pages, int max_prefix_len, float sm_scale, float* o_a,
                                  float* lse_a, void* workspace, size_t workspace_bytes,
                                  cpa_stream_t stream);

/*
 * Bytes of workspace cpa_prefill_hit needs for these sizes on the current
 * device (0 for sizes it would reject).
 */
size_t cpa_prefill_hit_workspace_size(int B, int N, int H_hit, int H_q, int H_kv, int head_dim,
                                      int page_size);

/*
 * Prefill after a prefix-cache hit ("Causal Attention ... KV hit area"
 * page): B requests of N tokens whose first H_hit tokens were cached; the
 * KV of all N tokens is already in the paged pool.  Suffix token i (absolute
 * position H_hit + i) attends keys 0..H_hit+i: the rectangle 0..H_hit-1 and
 * the causal triangle H_hit..H_hit+i, merged by the LSE identity.
 *   q           bf16 [B*M, H_q, head_dim], M = N - H_hit, token b*M + i
 *   page_table  int32 [B, pt_stride], pt_stride >= ceil(N / page_size)
 *   part        CPA_PREFILL_FULL (o bf16), CPA_PREFILL_RECT or
 *               CPA_PREFILL_TRI (o fp32: the piece alone, for checking)
 *   o, lse      [B*M, H_q, head_dim] and fp32 [B*M, H_q]
 * Supported: head_dim 128, page_size in {8,...,256}, 0 <= H_hit <= N.
 */
cpa_status cpa_prefill_hit(const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* page_table, int pt_stride, int B, int N, int H_hit,
                           int H_q, int H_kv, int head_dim, int page_size, int num_pages,
                           float sm_scale, int part, void* o, float* lse, void* workspace,
                           size_t workspace_bytes, cpa_stream_t stream);

/*
 * Bytes of workspace cpa_cascade_verify_shared needs for these sizes on the
 * current device (0 for sizes it would reject), for either of its schedules.
 * Besides the status word and merge scratch it holds the first level's fp32
 * partial result, B*topk*S*H_q*(head_dim + 1) floats.
 */
size_t cpa_cascade_verify_shared_workspace_size(int B, int n_groups, int topk, int S, int H_q,
                                                int H_kv, int head_dim, int page_size);

/*
 * Multi-level cascade verify.  Requests whose block tables begin with the
 * same physical pages share that prefix (KV-cache tutorial, block-table
 * example of section 5.3; share_prefix of section 6.2), e.g. one system
 * prompt for a whole batch.  The B requests form n_groups groups of
 * B/n_groups consecutive requests; each group has one shared prefix of
 * shared_len tokens, each request then its own prefix, each branch its own
 * drafts.  Draft s of branch k of request b sees the group's shared prefix,
 * request b's own prefix and drafts 0..s of branch k.  The shared prefix is
 * read from memory once per group:
 *   - shared_len a multiple of page_size: one launch of the fused cascade
 *     kernel; each request's prefix walk covers the group's shared pages and
 *     then its own, and the requests of a group, scheduled together, take the
 *     shared pages from L2 after the first read.
 *   - otherwise three levels merged by the cascade page's log-sum-exp
 *     identity: the shared prefix for all the group's draft queries at once
 *     (the tensor-core kernel in its rectangle mode, the group's queries as one
 *     block of suffix queries), then the own prefix once per request and the
 *     drafts once per branch (the fused cascade kernel), which merges.
 * Both give the same result up to rounding.
 *   shared_page_table  int32 [n_groups, shared_pt_stride]: the group's shared
 *                      pages; shared_pt_stride >= ceil(shared_len/page_size).
 *                      May be NULL when shared_len is 0.
 *   shared_len         host: shared prefix length of every group (>= 0).
 *   prefix_page_table, prefix_lens
 *                      each request's own prefix (the tokens after the shared
 *                      part), own position j at page row[j / page_size], slot
 *                      j % page_size; max_prefix_len bounds prefix_lens.
 *   other arguments    as for cpa_cascade_verify.
 * Supported: as for cpa_cascade_verify, and B a multiple of n_groups.
 */
cpa_status cpa_cascade_verify_shared(const void* q, const void* k_pages, const void* v_pages,
                                     const int32_t* shared_page_table, int shared_pt_stride,
                                     int n_groups, int shared_len,
                                     const int32_t* prefix_page_table, int prefix_pt_stride,
                                     const int32_t* draft_page_table, int draft_pt_stride,
                                     const int32_t* prefix_lens, int B, int topk, int S, int H_q,
                                     int H_kv, int head_dim, int page_size, int num_pages,
                                     int max_prefix_len, float sm_scale, void* o, float* lse,
                                     void* workspace, size_t workspace_bytes,
                                     cpa_stream_t stream);

/*
 * Bytes of workspace cpa_tree_verify needs for these sizes on the current
 * device (0 for sizes it would reject): the status word and the merge
 * scratch of the attention kernel.
 */
size_t cpa_tree_verify_workspace_size(int B, int N, int H_q, int H_kv, int head_dim,
                                      int page_size);

/*
 * Verify over general draft trees (KV-cache tutorial, section 8.2 tip box
 * on tree attention, and Q14): request b holds a prefix of L_b cached tokens
 * and a draft tree of N nodes, flattened so that every parent comes before
 * its children (BFS order does).  Node i attends the whole prefix and the
 * tree nodes of A(i), its ancestors and itself: the mask M[i, j] = 1 iff j is
 * in A(i), the tree generalisation of the causal mask.  The chain-per-branch
 * case of cpa_cascade_verify is the forest of topk chains.  One launch: the
 * tensor-core kernel reads the prefix once per request for all N nodes (the
 * cascade page's Pass A) and takes the N tree nodes as one more tile of the
 * same online softmax, masked per row by the node's ancestor mask (built on
 * chip from the parent array), so the two parts are merged there.
 *   q                  bf16 [B*N, H_q, head_dim]; token b*N + i is node i of
 *                      request b.
 *   tree_page_table    int32 [B, tree_pt_stride]: node j of request b's tree
 *                      is at logical position j (page j / page_size, slot
 *                      j % page_size); tree_pt_stride >= ceil(N / page_size).
 *   tree_parents       int32 [B, N] on the device: the BFS index of node i's
 *                      parent, or -1 for a root (a node whose parent is the
 *                      last prefix token; several roots make a forest).  Each
 *                      parent index must be below its node's; the device
 *                      sets CPA_DEV_BAD_TREE where it is not.
 *   other arguments    as for cpa_cascade_verify (topk = 1, S = N).
 *   o, lse             bf16 [B*N, H_q, head_dim], fp32 [B*N, H_q].
 * Supported: head_dim 128; 1 <= N <= CPA_MAX_TREE_NODES;
 * N*(H_q/H_kv) <= 256; page sizes as for cpa_cascade_verify.
 */
cpa_status cpa_tree_verify(const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* prefix_page_table, int prefix_pt_stride,
                           const int32_t* tree_page_table, int tree_pt_stride,
                           const int32_t* prefix_lens, const int32_t* tree_parents, int B, int N,
                           int H_q, int H_kv, int head_dim, int page_size, int num_pages,
                           int max_prefix_len, float sm_scale, void* o, float* lse,
                           void* workspace, size_t workspace_bytes, cpa_stream_t stream);

/*
 * The tree part of cpa_tree_verify alone: node i of request b against the
 * tree nodes of A(i) only.  One CTA per (request, KV head) stages that
 * head's N tree K/V rows in shared memory; a warp then serves one node and
 * up to 4 query heads of the group at a time.  q needs 8-byte alignment,
 * k_pages, v_pages and o_b 16-byte alignment.
 *   o_b   fp32 [B*N, H_q, head_dim];  lse_b fp32 [B*N, H_q].
 * Workspace: at least cpa_status_workspace_size() bytes (the status word).
 * Supported: head_dim 128; 1 <= N <= CPA_MAX_TREE_NODES.
 */
cpa_status cpa_tree_pass_b(const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* tree_page_table, int tree_pt_stride,
                           const int32_t* tree_parents, int B, int N, int H_q, int H_kv,
                           int head_dim, int page_size, int num_pages, float sm_scale,
                           float* o_b, float* lse_b, void* workspace, size_t workspace_bytes,
                           cpa_stream_t stream);

/*
 * Read the device status word of `workspace` (written by the last call that
 * used it) into *status_out (host).  SYNCHRONISES `stream`.  Returns CPA_OK
 * when the word is 0, otherwise the status matching its most serious bit
 * (TIMEOUT, then BAD_PAGE, then BAD_LENGTH, then BAD_TREE).
 */
cpa_status cpa_get_device_status(const void* workspace, uint32_t* status_out,
                                  cpa_stream_t stream);

/*
 * Failure-detection check: launch one kernel that waits on a barrier nothing
 * will ever complete, with a wait limit of `limit_us` microseconds, so the
 * kernel gives up, sets CPA_DEV_TIMEOUT in the workspace status word and
 * returns.  Used by tests to exercise the bounded-wait path without hanging
 * the GPU.  Workspace: cpa_status_workspace_size() bytes.
 */
cpa_status cpa_debug_wait_timeout(void* workspace, size_t workspace_bytes, int limit_us,
                                  cpa_stream_t stream);

/*
 * Host-side view of the work partition the attention kernels use, for
 * tests: `total` tiles split over `n_ctas` CTAs, CTA c owning
 * [begin, end).  Returns the owner CTA of tile `tile` and fills begin/end
 * of CTA `cta` (host pointers).  Returns -1 on bad arguments, and -2 if the
 * two forms of the split arithmetic the kernels use (64-bit division, and
 * 32-bit division where total * n_ctas < 2^31) disagree, which they must not.
 */
int cpa_plan_partition(int64_t total, int n_ctas, int cta, int64_t tile, int64_t* begin,
                       int64_t* end);

/*
 * Static-scratch cascade verify: the same computation, arguments and
 * results as cpa_cascade_verify, but no workspace argument and no
 * allocation by anyone.  The source pages have no counterpart of this call;
 * it exists for callers that cannot call cudaMalloc.  Examples: an inference
 * engine that reserves nearly all HBM for its paged KV pool at start-up and
 * forbids later driver allocations (they would fail or fragment the pool);
 * a latency-critical decode loop that cannot pay for cudaMalloc's implicit
 * device-wide synchronisation; plugin code hosted by a framework that owns
 * every device buffer and hands the plugin no allocator.
 *
 * Scratch: a file-scope device array of CPA_STATIC_SCRATCH_BYTES, which every
 * GPU that loads this library holds until the process exits.  The scratch a
 * call needs is a fixed part that grows with the device's SM count (two fp32
 * partial-result slots of 256 rows x 128 columns per SM, about 262 KB per SM,
 * 40 MB on 152 SMs) plus 4 bytes per (request, KV head).  Sizes that need
 * more than the array are rejected with CPA_ERR_WORKSPACE before anything
 * is launched; so the usable shapes shrink as the SM count grows, and on a
 * part with more than about 180 SMs no shape fits.  Other invalid arguments
 * get the same status codes as cpa_cascade_verify.
 *
 * The first call on a device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress); make that first call
 * before any stream capture.  All calls on a device share the one array and
 * it keeps the last call's contents: each call clears the status word and
 * merge counters it needs (asynchronous memset on `stream`) before its
 * kernel runs.  Calls that overlap on the GPU (different streams, no
 * ordering between them) race on the array.
 *
 * Errors only the GPU can see (bad page id, bad prefix length, wait timeout)
 * go to the status word at the start of the array; read it with
 * cpa_noalloc_device_status.
 */
#define CPA_STATIC_SCRATCH_BYTES (48u * 1024u * 1024u)

cpa_status cpa_cascade_verify_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                      const int32_t* prefix_page_table, int prefix_pt_stride,
                                      const int32_t* draft_page_table, int draft_pt_stride,
                                      const int32_t* prefix_lens, int B, int topk, int S, int H_q,
                                      int H_kv, int head_dim, int page_size, int num_pages,
                                      int max_prefix_len, float sm_scale, void* o, float* lse,
                                      cpa_stream_t stream);

/*
 * The device status word of the static scratch of the current device, as
 * written by the last cpa_cascade_verify_noalloc call on it, into
 * *status_out (host).  Same return values as cpa_get_device_status, and
 * like it SYNCHRONISES `stream`.  The source pages have no counterpart of
 * this call either.
 */
cpa_status cpa_noalloc_device_status(uint32_t* status_out, cpa_stream_t stream);

/* Library version, e.g. 100 for 0.1.0. */
int cpa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CPA_H_ */
