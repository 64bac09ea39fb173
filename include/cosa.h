/*
 * cosa.h - C ABI of libcosa: CoSA block-sparse long-context prefill on GB300 (sm_103a).
 *
 * Two calls make up the prefill attention of one layer:
 *
 *   cosa_proxy_select   the Kernel-Aware Proxy (KAP).  CoSA: "Accelerating Long-Context
 *                       Inference via Proxy-Kernel Co-Designed Sparse Attention",
 *                       Sec. 4.2, Eqs. (8)-(14), Algorithm A (proxy stage).  Scores each
 *                       (query block, key block) pair from stride-sampled queries and
 *                       keys, flags the blocks that hold a sampled row's maximum (HRM),
 *                       and writes the computation-order mask M_KAP: per query block,
 *                       the HRM blocks then the rest, each by descending score, cut to
 *                       the stage-1 budget.
 *
 *   cosa_sparse_prefill the Ordered-Skipping Kernel (OSK).  Same paper, Sec. 4.3 and
 *                       Algorithm A (ordered-skipping stage): per query block, visits the
 *                       mask's blocks in order through the page table, keeps the exact
 *                       running row maximum, skips a block when every row's local maximum
 *                       is more than ln(N/Delta) below its running maximum (Eq. (5)), and
 *                       accumulates exact online softmax over the rest.  The output of
 *                       each query is the softmax-weighted sum over its token set as the
 *                       PageWeaver notes define it (Sec. 2.1, Eqs. (1)-(2)): tokens of
 *                       computed blocks, below the request length, not after the query;
 *                       invalid or repeated block IDs add nothing; no support gives 0.
 *
 * Conventions shared by every call
 *   - Every pointer argument is DEVICE memory owned by the caller, except `p` (host).
 *     The library allocates nothing, keeps no pointer after a call returns, and
 *     enqueues all work on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream).  Calls are asynchronous; outputs are valid after the stream reaches them.
 *   - Tensors are dense, row-major, 16-byte aligned:
 *       q           bf16 [total_tokens, Hq, d]          requests packed by cu_seqlens
 *       k_cache     bf16 [num_pages, P, Hkv, d]         paged keys (PagedAttention layout)
 *       v_cache     bf16 [num_pages, P, Hkv, d]
 *       page_table  int32 [num_reqs, max_pages_per_req] logical page -> physical page
 *       cu_seqlens  int32 [num_reqs + 1]                cu_seqlens[0] = 0, non-decreasing
 *       mask        int32 [num_reqs, Hq, nqb_max, mask_pitch]   block IDs, -1 padded
 *       mask_len    int32 [num_reqs, Hq, nqb_max]                entries used per row
 *       out         bf16 [total_tokens, Hq, d]
 *     with nqb_max = ceil(max_seqlen / block_size).  Query head h reads kv head
 *     h / (Hq / Hkv).  Logical block j of a request covers tokens [j*b, (j+1)*b) and
 *     pages j*b/P .. (j+1)*b/P - 1 of its page-table row.
 *   - A page-table entry outside [0, num_pages) means the page does not exist: its
 *     tokens take part in nothing and are never read.  Mask entries < 0, > i (after the
 *     query block), >= ceil(L/b), and repeats of an earlier entry of the same row are
 *     ignored and never dereferenced.  K/V values must be finite in every slot of every
 *     page a mask references (slots past the request length included).
 *   - Return value: COSA_OK, or a negative status for an error found on the host before
 *     anything is enqueued (COSA_ERR_INVALID_ARG, COSA_ERR_UNSUPPORTED, COSA_ERR_WORKSPACE)
 *     or a failed launch (COSA_ERR_CUDA).  Errors found on the device are written to
 *     *device_status (an int32 the caller zeroes; may be NULL): COSA_ERR_DEVICE_TIMEOUT
 *     when a bounded wait inside a kernel ran out (the kernel then stops cleanly and the
 *     outputs are undefined), COSA_ERR_BAD_INPUT when cu_seqlens disagree with `p`.
 */
#ifndef COSA_H_
#define COSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define COSA_OK 0
#define COSA_ERR_INVALID_ARG (-1)
#define COSA_ERR_UNSUPPORTED (-2)
#define COSA_ERR_CUDA (-3)
#define COSA_ERR_DEVICE_TIMEOUT (-4)
#define COSA_ERR_WORKSPACE (-5)
#define COSA_ERR_BAD_INPUT (-6)

/* cosa_params.flags */
#define COSA_FLAG_NONE 0
/* Test hook for the bounded waits (cosa_sparse_prefill only): the producer of K and Q tiles issues
   nothing, so every wait inside the kernel runs out after its 2 s budget, the kernel stops cleanly and
   *device_status becomes COSA_ERR_DEVICE_TIMEOUT; out is then undefined.  The CUDA context stays usable. */
#define COSA_FLAG_TEST_STALL 1
/* Ablation switch of cosa_proxy_select (ignored by cosa_sparse_prefill): write the same K_i selected
   blocks in ascending block order instead of the computation order rho_i of Eq. (14), i.e. visiting
   without KV page remapping (the no-remapping arm of the paper's Sec. 5.4, Fig. 6 and App. D.4). */
#define COSA_FLAG_ASCENDING_ORDER 2
/* Ablation switch of cosa_sparse_prefill (ignored by cosa_proxy_select): read each mask row as the
   binary block mask M_01 of the paper's Eq. (3) instead of a list of block IDs.  Entry j != 0 selects
   key block j.  The kernel walks every block j < min(mask_len, i + 1) in ascending order and drops the
   unselected ones by a logical test, each still taking one turn through its pipeline (the logical
   mask skipping of BSA kernels, Sec. 4.3 and App. D.3); visit_flags[j] reports block j, and
   entries past the walk are IGNORED.  The output equals that of the ascending ID list of the selected
   blocks. */
#define COSA_FLAG_BINARY_MASK 4
/* Stage-1 budget by top-p (cosa_proxy_select; the paper's Sec. 5.1 and App. D.1 use p = 0.95): budget_ppm
   holds p in parts per million and K_i is the length of the shortest prefix of rho_i (Eq. (13)) whose
   block scores s_ij (Eq. (11)) sum to at least p times the sum over all causal candidates j <= i.  The
   length is certified from the error bounds of the fp32 scores; where those bounds leave it open, it is
   taken from scores of every candidate evaluated at float64 accuracy.  mask_pitch must be >=
   ceil(max_seqlen / block_size), since K_i can reach i + 1. */
#define COSA_FLAG_TOP_P 8
/* GQA page union (cosa_sparse_prefill; ignored by cosa_proxy_select).  PageWeaver notes, Sec. 2.2: the
   query heads of a kv group select largely the same pages, so one K load can serve several of them
   (the union U_G with a membership mask per head).  Under this flag one CTA serves two query heads
   2x, 2x+1 of a kv group (the last head alone when Hq/Hkv is odd) for one query block, from one
   stream of K tiles: the two heads' de-duplicated valid block lists, each in its own mask order, are
   merged by taking at every step the block that is next for both heads if they agree, else the
   lower of the two next block IDs (which serves only the head it is next for).  Each head still
   visits exactly its own blocks in its own order with its own running maximum and skip vote, so
   out and the visit decisions equal those of the default kernel bit for bit; visit_flags entries
   whose K tile was loaded once for both heads carry COSA_VISIT_SHARED_LOAD in addition.  Requires
   block_size 128; not combinable with COSA_FLAG_BINARY_MASK. */
#define COSA_FLAG_GQA_UNION 16

/* values written to visit_flags (one per mask entry) */
#define COSA_VISIT_COMPUTED 0 /* softmax and P.V accumulated (pattern 3 of the paper's Fig. 4) */
#define COSA_VISIT_SKIPPED 1  /* Q.K^T computed, in-kernel skip rule fired (pattern 2)         */
#define COSA_VISIT_IGNORED 2  /* invalid, repeated, or past mask_len: never loaded            */
#define COSA_VISIT_SHARED_LOAD 4 /* bit OR-ed onto COMPUTED / SKIPPED under COSA_FLAG_GQA_UNION:
                                    the block's K tile was gathered once for both heads of a pair */

typedef struct cosa_params {
  int32_t num_reqs;          /* B >= 1                                                        */
  int32_t num_q_heads;       /* Hq >= 1                                                       */
  int32_t num_kv_heads;      /* Hkv >= 1, Hq % Hkv == 0                                       */
  int32_t head_dim;          /* d: 64 or 128                                                  */
  int32_t block_size;        /* b: 64 or 128 (query and key block)                           */
  int32_t page_size;         /* P: 16, 32, 64 or 128, with b % P == 0                          */
  int32_t stride;            /* s: KAP sampling stride, b % s == 0, b / s in {4, 8, 16}       */
  int32_t total_tokens;      /* T = cu_seqlens[B]                                             */
  int32_t max_seqlen;        /* >= every request length L_b; sizes grids and mask rows        */
  int32_t num_pages;         /* rows of k_cache / v_cache                                     */
  int32_t max_pages_per_req; /* page-table row pitch, >= ceil(max_seqlen / P)                 */
  int32_t mask_pitch;        /* Kmax: mask row pitch (entries per query block)                */
  int32_t budget_ppm;        /* stage-1 fraction B1 in parts per million, 1..1000000:
                                K_i = ceil(B1 * (i + 1)), i the query block (0-based); with
                                COSA_FLAG_TOP_P the top-p threshold p instead                   */
  int32_t flags;             /* COSA_FLAG_*                                                   */
  double sm_scale;           /* logit scale, normally 1/sqrt(d)                                */
  double skip_delta;         /* Delta of the skip threshold ln(Delta / L_b); <= 0 disables
                                in-kernel skipping (paper App. D.1: Delta = -1)                */
} cosa_params;

/* Library version, (major << 16) | minor. */
int cosa_version(void);

/* Human-readable text for a status code; never NULL. */
const char* cosa_status_string(int status);

/*
 * KAP: write the computation-order mask (CoSA Sec. 4.2, Eqs. (8)-(14); Algorithm A, proxy stage).
 *
 *   q, cu_seqlens, k_cache, page_table   inputs as above (V is not read)
 *   mask       out: for every request b, head h and query block i < ceil(L_b / b):
 *              mask[b,h,i,0:K_i] = the ordered block IDs, mask[b,h,i,K_i:mask_pitch] = -1,
 *              with K_i = ceil(budget_ppm * (i+1) / 1e6), or the top-p length (COSA_FLAG_TOP_P).
 *              Rows of absent query blocks (i >= ceil(L_b / b)) are set to -1.  Requires
 *              mask_pitch >= K_i for all i.
 *   mask_len   out: K_i per row (0 for absent query blocks).
 *   workspace  scratch of at least cosa_proxy_workspace_size(p) bytes (256-byte aligned);
 *              its content on entry does not matter and is undefined on exit.
 *
 * Selections are exact: the fp32 tensor-core scores carry error bounds, and every
 * order or cut (fraction or top-p) they cannot certify is settled with logits at
 * float64 accuracy or better, so the mask equals the one computed from exact
 * real-number scores except where two scores, or a prefix mass and p times the total,
 * agree to within float64 rounding.  Stride sampling keeps token positions 0, s, 2s,
 * ...; ties in score go to the lower block ID.
 */
/* Bytes of workspace cosa_proxy_select needs for `p`; 0 if cosa_proxy_select would refuse `p`. */
size_t cosa_proxy_workspace_size(const cosa_params* p);
int cosa_proxy_select(const cosa_params* p, const void* q, const int32_t* cu_seqlens, const void* k_cache,
                      const int32_t* page_table, int32_t* mask, int32_t* mask_len, void* workspace,
                      size_t workspace_bytes, int32_t* device_status, void* stream);

/*
 * KAP without a workspace argument, for callers that cannot allocate device memory.  (The
 * paper has no counterpart; this is a deployment variant of cosa_proxy_select.)
 *
 * Some callers cannot call cudaMalloc or hand out a scratch buffer: code running inside a
 * host framework that owns all device memory through its own allocator and exposes none to
 * plug-ins, or a serving loop that must not enter an allocator while requests are in flight
 * (allocation can block, synchronize the device, or fail once a pool has reserved most of
 * HBM).  This entry point takes the same arguments as cosa_proxy_select minus the workspace
 * and computes the same mask.  Its scratch is a fixed array of COSA_STATIC_SCRATCH_BYTES
 * inside the library: every GPU that loads the library holds that much device memory until
 * the process exits, and the call itself allocates nothing.
 *
 *   - Size limit: a problem whose cosa_proxy_workspace_size(p) exceeds COSA_STATIC_SCRATCH_BYTES
 *     is rejected with COSA_ERR_WORKSPACE before anything is enqueued.
 *   - The first call in a CUDA context (normally the device's primary context) looks up the
 *     array's device address with that device current (a runtime call that does not allocate)
 *     and keeps it for that context; make that first call before any stream capture begins on
 *     that device.  A context created later (after cudaDeviceReset, or another context made
 *     current through the driver API) gets its own lookup on its first call.
 *   - Invalid parameters are refused exactly as cosa_proxy_select refuses them.
 *   - Every call shares the one array and leaves its contents behind; the kernels initialise
 *     everything they read.  Calls whose work overlaps on the GPU (different streams, or
 *     several host threads on one device) race on the array: order them on one stream.
 */
#define COSA_STATIC_SCRATCH_BYTES ((size_t)64 << 20)
int cosa_proxy_select_static(const cosa_params* p, const void* q, const int32_t* cu_seqlens, const void* k_cache,
                             const int32_t* page_table, int32_t* mask, int32_t* mask_len, int32_t* device_status,
                             void* stream);

/*
 * OSK: ordered-skipping sparse prefill (CoSA Sec. 4.3; Algorithm A (ordered-skipping stage)).
 *
 *   mask, mask_len  the visiting order per (request, head, query block); rows may hold
 *                   any IDs (see the conventions above).  Entries k < mask_len are visited
 *                   in order; mask_len is clamped to mask_pitch.
 *   out             out: attention output for every token of every request (bf16,
 *                   round-to-nearest-even from fp32 accumulators).
 *   visit_flags     optional out (NULL to skip): uint8 [B, Hq, nqb_max, mask_pitch],
 *                   COSA_VISIT_* per mask entry; entries at k >= mask_len are IGNORED.
 *   workspace       scratch of at least cosa_prefill_workspace_size(p) bytes (may be 0).
 *
 * The skip threshold of request b is ln(skip_delta / L_b); with skip_delta <= 0 every
 * valid block is computed.  A block is skipped when every row of the query block that
 * exists satisfies m_loc - m < threshold, m being the running maximum after the block
 * (rows with no visible key in the block agree to skip).
 */
size_t cosa_prefill_workspace_size(const cosa_params* p);
int cosa_sparse_prefill(const cosa_params* p, const void* q, const int32_t* cu_seqlens, const void* k_cache,
                        const void* v_cache, const int32_t* page_table, const int32_t* mask,
                        const int32_t* mask_len, void* out, uint8_t* visit_flags, void* workspace,
                        size_t workspace_bytes, int32_t* device_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* COSA_H_ */
