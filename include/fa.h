/*
 * fa.h -- C ABI of the GB300 (sm_103a) fused attention forward library.
 *
 * What is computed (FlashAttn operator guide, functional description;
 * aclnnIncreFlashAttention guide §1.2):
 *
 *     out = softmax(scale * Q K^T  [masked]) V,   lse = log sum_j exp(scale * q.k_j)
 *
 * row by row, tile by tile with a running max m and sum l, so the
 * S_q x S_kv score matrix is never stored (FlashAttn guide, functional
 * description and developer guide §3). Two regimes:
 *   - prefill (fa_forward): S_q = S_kv rows, optional causal mask, optional
 *     per-key mask, GQA;
 *   - decode (fa_decode): S_q = 1 against a padded KV cache with per-batch
 *     actual lengths, split along the keys into chunks (Split-KV) whose
 *     partial results are merged by their log-sum-exp (FlashAttn guide §1.9
 *     and §10; aclnnIncreFlashAttention guide §8.2-§8.3; FlashDecoding
 *     tutorial §二-§三).
 *
 * Conventions shared by every entry point
 *   - Tensors q, k, v, out are bf16, dense (contiguous), in one of two
 *     layouts (FlashAttn guide, parameter layouts; aclnnIncreFlashAttention
 *     guide §四 inputLayout): BNSD = [B, N, S, D] or BSND = [B, S, N, D]
 *     (BSH is BSND memory). out has the shape and layout of q. The base
 *     address of every tensor must be 16-byte aligned.
 *   - lse (optional, may be NULL) is fp32 [B, num_heads, S_q], natural log
 *     (FlashAttn guide §1.6).
 *   - GQA: num_heads must be a multiple of num_kv_heads; query head h reads
 *     KV head h / (num_heads / num_kv_heads) (FlashAttn guide §1.1).
 *     num_kv_heads == 0 means num_kv_heads = num_heads
 *     (aclnnIncreFlashAttention guide §四, numKeyValueHeads).
 *   - key_mask (optional, may be NULL): device uint8 [B, S_kv], one flag per
 *     key shared by all heads and query rows; nonzero = the key is excluded
 *     (aclnnIncreFlashAttention guide §8.1: true positions are masked out).
 *   - actual_seq_lengths: HOST int64 [B], valid KV length per batch; keys at
 *     or past it are ignored entirely and may hold any bits, NaN included
 *     (aclnnIncreFlashAttention guide §四 actualSeqLengths and §1.1).
 *   - A query row with no valid key gets out = 0 and lse = +inf (FlashAttn
 *     guide §1.7, row invalid).
 *   - Head dimension D must be 64, 128 or 256 (FlashAttn guide §3 lists
 *     D in {64, 128, 256}).
 *   - Two-stage use as in aclnnIncreFlashAttention guide §三: ask for the
 *     workspace size, allocate it on the device, then call. The caller owns
 *     every buffer; the library allocates no device memory and keeps no
 *     pointer after a call returns.
 *   - All device work is enqueued on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and runs asynchronously. Argument errors are
 *     detected and returned before anything is enqueued.
 *   - Results are deterministic: every reduction runs in a fixed order (in
 *     decode, atomic counters only decide which CTA merges a sequence's pieces,
 *     not the order in which they are summed).
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FA_ABI_VERSION 1

/* Status codes; the classes follow aclnnIncreFlashAttention guide §四
 * (return values: null pointer, invalid parameter, runtime error). */
typedef enum {
  FA_OK = 0,
  FA_ERR_NULLPTR = 1,             /* a required pointer is NULL */
  FA_ERR_PARAM_INVALID = 2,       /* a size, layout, mode or length is outside the contract */
  FA_ERR_UNSUPPORTED = 3,         /* allowed by the pages but not built here (D not 64/128/256) */
  FA_ERR_WORKSPACE_TOO_SMALL = 4, /* workspace_bytes below the size query's answer */
  FA_ERR_RUNTIME = 5,             /* a CUDA call failed (launch, copy, device query) */
  FA_ERR_DEVICE_TIMEOUT = 6,      /* a kernel's bounded wait expired; outputs are undefined */
  FA_ERR_DEVICE_CHECK = 7         /* debug builds only (libfa_gb300_debug.so, FA_DEBUG): a
                                     device-side index check failed and the access was skipped */
} fa_status;

typedef enum {
  FA_LAYOUT_BNSD = 0,
  FA_LAYOUT_BSND = 1,
  /* paged K/V caches (FlashAttn guide §1.2, layout_kv): fa_decode_paged, fa_forward_paged */
  FA_LAYOUT_PA_BBND = 2, /* [num_blocks, block_size, KV_N, D]: rows of a block as BSND */
  FA_LAYOUT_PA_BNBD = 3  /* [num_blocks, KV_N, block_size, D]: rows of a block as BNSD */
} fa_layout;

/* Mask modes, numbered as in FlashAttn guide §1.5 (0 = none, 3 = causal,
 * 4 = window; the window takes its widths through fa_forward_window). */
typedef enum { FA_MASK_NONE = 0, FA_MASK_CAUSAL = 3, FA_MASK_WINDOW = 4 } fa_mask_mode;

/* Version of this ABI (FA_ABI_VERSION). */
int fa_abi_version(void);

/* Static text for a status code; never NULL. */
const char* fa_status_string(int status);

/* ---------------------------------------------------------------- prefill
 * Workspace bytes fa_forward needs for these sizes (>= 256; holds the
 * device status word and, when a key mask or lengths are given, a per-tile
 * key-validity table). Pure host arithmetic; 0 when a size is negative. */
size_t fa_forward_workspace_size(int64_t B, int64_t S_q, int64_t S_kv, int64_t num_heads,
                                 int64_t num_kv_heads, int64_t D);

/* Fused attention forward (prefill).
 *   q    [B, num_heads, S_q, D] (BNSD) or [B, S_q, num_heads, D] (BSND), device bf16
 *   k, v [B, num_kv_heads, S_kv, D] or [B, S_kv, num_kv_heads, D], device bf16
 *   mask_mode           FA_MASK_NONE or FA_MASK_CAUSAL; causal keeps key j for
 *                       query row i iff j <= i and requires S_q == S_kv
 *   key_mask            NULL or device uint8 [B, S_kv] (nonzero = excluded)
 *   actual_seq_lengths  NULL or HOST int64 [B], each in [0, S_kv]
 *   scale               multiplies Q K^T before the softmax (finite)
 *   out                 device bf16, shape and layout of q
 *   lse                 NULL or device fp32 [B, num_heads, S_q]
 *   workspace           device, >= fa_forward_workspace_size(...) bytes,
 *                       256-byte aligned; contents need no initialisation
 * B == 0 or S_q == 0 is a no-op returning FA_OK. S_kv == 0 makes every row
 * invalid (out 0, lse +inf). */
fa_status fa_forward(const void* q, const void* k, const void* v, int mask_mode,
                     const uint8_t* key_mask, const int64_t* actual_seq_lengths, int64_t B,
                     int64_t S_q, int64_t S_kv, int64_t num_heads, int64_t num_kv_heads,
                     int64_t D, float scale, int layout, void* out, float* lse,
                     void* workspace, size_t workspace_bytes, void* stream);

/* fa_forward with K and V in a paged cache (FlashAttn guide §1.2: layout_kv
 * PA_BBND / PA_BNBD, usable with the q layouts BSND and BNSD): blocks of
 * block_size key rows in a pool, and a block table per sequence.
 *   k_cache, v_cache  device bf16 pools, kv_layout FA_LAYOUT_PA_BBND
 *                     [num_blocks, block_size, num_kv_heads, D] or
 *                     FA_LAYOUT_PA_BNBD [num_blocks, num_kv_heads, block_size, D]
 *   block_table       device int32 [B, max_blocks_per_seq]: key row r of
 *                     sequence b is row r % block_size of block
 *                     block_table[b * max_blocks_per_seq + r / block_size]
 *   block_size        a multiple of 16 in [16, 1024]
 *   max_blocks_per_seq  * block_size >= S_kv (the table covers every key row)
 *   S_kv              the keys of each sequence (its logical length); the
 *                     other arguments (q and out in `layout`, mask_mode,
 *                     key_mask [B, S_kv], actual_seq_lengths, lse, the
 *                     workspace of fa_forward_workspace_size) as in fa_forward
 * Entries of a table past the blocks a sequence's keys use may hold any value:
 * a KV tile that reaches past the last key may load rows through them (an id
 * outside [0, num_blocks) loads zeros), and those keys are excluded before
 * any product, with their V rows zeroed.
 * Errors: block_table NULL with B > 0 -> FA_ERR_NULLPTR; an unknown
 * kv_layout, a bad block_size or a table too short for S_kv ->
 * FA_ERR_PARAM_INVALID; otherwise those of fa_forward. */
fa_status fa_forward_paged(const void* q, const void* k_cache, const void* v_cache, int kv_layout,
                           const int32_t* block_table, int64_t max_blocks_per_seq,
                           int64_t num_blocks, int64_t block_size, int mask_mode,
                           const uint8_t* key_mask, const int64_t* actual_seq_lengths, int64_t B,
                           int64_t S_q, int64_t S_kv, int64_t num_heads, int64_t num_kv_heads,
                           int64_t D, float scale, int layout, void* out, float* lse,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Fused attention forward over packed variable-length sequences (the TND
 * layout of FlashAttn guide §1.3 and §1.4: the tokens of all sequences laid
 * end to end, cu_seqlens giving each sequence's start).
 *   q, out   [T_q, num_heads, D], device bf16, T_q = cu_seqlens_q[B]
 *   k, v     [T_kv, num_kv_heads, D], device bf16, T_kv = cu_seqlens_kv[B]
 *   cu_seqlens_q, cu_seqlens_kv  HOST int64 [B + 1], 0 first, non-decreasing;
 *            sequence b is q rows [cu_q[b], cu_q[b+1]) against k/v rows
 *            [cu_kv[b], cu_kv[b+1]); a sequence with no keys gives out 0,
 *            lse +inf; one with no queries writes nothing
 *   mask_mode  FA_MASK_NONE or FA_MASK_CAUSAL (causal needs equal q and kv
 *            lengths per sequence, top-left aligned within it)
 *   lse      NULL or device fp32 [T_q, num_heads]
 *   workspace  >= fa_forward_varlen_workspace_size(B, longest q sequence,
 *            longest kv sequence, ...) bytes, 256-byte aligned
 * Errors: bad offsets or lengths -> FA_ERR_PARAM_INVALID; NULL offsets ->
 * FA_ERR_NULLPTR; otherwise those of fa_forward. */
size_t fa_forward_varlen_workspace_size(int64_t B, int64_t max_seqlen_q, int64_t max_seqlen_kv,
                                        int64_t num_heads, int64_t num_kv_heads, int64_t D);
fa_status fa_forward_varlen(const void* q, const void* k, const void* v,
                            const int64_t* cu_seqlens_q, const int64_t* cu_seqlens_kv,
                            int mask_mode, int64_t B, int64_t num_heads, int64_t num_kv_heads,
                            int64_t D, float scale, void* out, float* lse, void* workspace,
                            size_t workspace_bytes, void* stream);

/* fa_forward_varlen with a sliding window (FlashAttn guide §1.5, mask_mode 4)
 * inside every packed sequence: query row i of a sequence keeps key j of the
 * same sequence iff
 *     (win_left  < 0 or j >= i - win_left) and (win_right < 0 or j <= i + win_right),
 * i and j counted from the sequence's first token (top-left aligned, so
 * (-1, 0) is causal and (-1, -1) no mask). A window needs equal q and kv
 * lengths per sequence; widths below -1 are FA_ERR_PARAM_INVALID. KV tiles
 * wholly outside every row's window are never loaded or multiplied. The
 * workspace (fa_forward_varlen_workspace_size) and the other errors are those
 * of fa_forward_varlen. */
fa_status fa_forward_varlen_window(const void* q, const void* k, const void* v,
                                   const int64_t* cu_seqlens_q, const int64_t* cu_seqlens_kv,
                                   int64_t win_left, int64_t win_right, int64_t B,
                                   int64_t num_heads, int64_t num_kv_heads, int64_t D, float scale,
                                   void* out, float* lse, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* The packed-sequence forward with every option of FlashAttn guide §1.3-§1.5
 * at once: the used lengths of §1.4 and a key mask, with causal or a window.
 *   seqused_q, seqused_kv  NULL or HOST int64 [B], each >= 0: sequence b uses
 *            the first min(cu_q[b+1] - cu_q[b], seqused_q[b]) query rows and
 *            the first min(cu_kv[b+1] - cu_kv[b], seqused_kv[b]) keys of its
 *            span (when both are given the shorter length holds, §1.4). Keys
 *            past the used kv length are ignored whatever they hold; query
 *            rows past the used q length are truncated rows: out 0, lse +inf
 *            (§1.7 counts seqused truncation among the causes of a row with
 *            no valid key)
 *   key_mask NULL or device uint8 [T_kv], one flag per packed key row
 *            (nonzero = excluded), shared by all heads and query rows
 *   win_left, win_right  the window of fa_forward_varlen_window: (-1, -1) no
 *            mask, (-1, 0) causal; causal and windows need equal q and kv
 *            spans per sequence (cu_seqlens), top-left aligned within it
 * The other arguments, the workspace (fa_forward_varlen_workspace_size with
 * the longest spans) and the errors are those of fa_forward_varlen; a
 * negative seqused entry is FA_ERR_PARAM_INVALID. */
fa_status fa_forward_varlen_ex(const void* q, const void* k, const void* v,
                               const int64_t* cu_seqlens_q, const int64_t* cu_seqlens_kv,
                               const int64_t* seqused_q, const int64_t* seqused_kv,
                               const uint8_t* key_mask, int64_t win_left, int64_t win_right,
                               int64_t B, int64_t num_heads, int64_t num_kv_heads, int64_t D,
                               float scale, void* out, float* lse, void* workspace,
                               size_t workspace_bytes, void* stream);

/* Fused attention forward with a sliding window (FlashAttn guide §1.5,
 * mask_mode 4: a band of win_left tokens before and win_right tokens after
 * each query). Query row i keeps key j iff
 *     (win_left  < 0 or j >= i - win_left) and (win_right < 0 or j <= i + win_right),
 * top-left aligned as causal is; -1 means no limit on that side, so (-1, 0)
 * is causal and (-1, -1) no mask. A window requires S_q == S_kv; widths below
 * -1 are FA_ERR_PARAM_INVALID. KV tiles wholly outside every row's window
 * are never loaded or multiplied. All other arguments, the workspace
 * (fa_forward_workspace_size) and the errors are those of fa_forward. */
fa_status fa_forward_window(const void* q, const void* k, const void* v, int64_t win_left,
                            int64_t win_right, const uint8_t* key_mask,
                            const int64_t* actual_seq_lengths, int64_t B, int64_t S_q,
                            int64_t S_kv, int64_t num_heads, int64_t num_kv_heads, int64_t D,
                            float scale, int layout, void* out, float* lse, void* workspace,
                            size_t workspace_bytes, void* stream);

/* ----------------------------------------------------------------- decode
 * Workspace bytes fa_decode needs. num_splits as for fa_decode (0 = the
 * split heuristic; the answer then covers any choice it can make).
 * Pure host arithmetic; 0 when an argument is out of range. */
size_t fa_decode_workspace_size(int64_t B, int64_t S_kv_max, int64_t num_heads,
                                int64_t num_kv_heads, int64_t D, int num_splits);

/* Incremental (decode) attention with Split-KV.
 *   q    [B, num_heads, 1, D] (BNSD) or [B, 1, num_heads, D] (BSND): the same
 *        memory either way, device bf16
 *   k, v padded caches [B, num_kv_heads, S_kv_max, D] or [B, S_kv_max, num_kv_heads, D]
 *   key_mask            NULL or device uint8 [B, S_kv_max] (nonzero = excluded)
 *   actual_seq_lengths  HOST int64 [B], required, each in [0, S_kv_max]
 *   num_splits          0: one equal share of all K/V rows per SM (see
 *                       fa_decode_plan); n > 0: shares of ceil(S_kv_max / n)
 *                       rows rounded up to a multiple of 64, so a
 *                       full-length sequence is cut into about n pieces
 *   out                 device bf16 [B, num_heads, D] (either layout)
 *   lse                 NULL or device fp32 [B, num_heads]
 *   workspace           device, >= fa_decode_workspace_size(..., num_splits)
 *                       bytes, 256-byte aligned
 * The lengths are read on the host during the call. On `stream` the call
 * clears the status word and the per-sequence piece counters at the start of
 * the workspace, copies the lengths' prefix sums there when B > 1024 (else
 * they travel in the launch parameters), and launches one kernel: the CTA
 * that finishes the last piece of a sequence cut into several merges them. */
fa_status fa_decode(const void* q, const void* k, const void* v, const uint8_t* key_mask,
                    const int64_t* actual_seq_lengths, int64_t B, int64_t S_kv_max,
                    int64_t num_heads, int64_t num_kv_heads, int64_t D, float scale, int layout,
                    int num_splits, void* out, float* lse, void* workspace,
                    size_t workspace_bytes, void* stream);

/* Layouts of the decode key mask (aclnnIncreFlashAttention guide §四,
 * attenMask): one flag per key shared by every query head, (B, 1, 1, S) =
 * [B, S_kv_max]; or one row of flags per query head, (B, N, 1, S) =
 * [B, num_heads, S_kv_max], or the same rows for every batch, (1, N, 1, S) =
 * [num_heads, S_kv_max]. */
typedef enum {
  FA_KEY_MASK_B11S = 0,
  FA_KEY_MASK_BN1S = 1,
  FA_KEY_MASK_1N1S = 2
} fa_key_mask_layout;

/* fa_decode with the key mask in any of the layouts above (fa_decode's
 * key_mask is FA_KEY_MASK_B11S). With a per-head mask, query head h keeps
 * key j iff j < actual_seq_lengths[b] and its own flag is 0; a key that some
 * head of its KV group still sees must hold finite K and V values (keys past
 * a length, or masked for every head of the group, may hold anything).
 * key_mask_layout outside the enum -> FA_ERR_PARAM_INVALID; the other
 * arguments, the workspace and the errors are those of fa_decode. */
fa_status fa_decode_masked(const void* q, const void* k, const void* v, const uint8_t* key_mask,
                           int key_mask_layout, const int64_t* actual_seq_lengths, int64_t B,
                           int64_t S_kv_max, int64_t num_heads, int64_t num_kv_heads, int64_t D,
                           float scale, int layout, int num_splits, void* out, float* lse,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Split-KV decode against a paged K/V cache (FlashAttn guide §1.2,
 * PagedAttention: the cache is stored in blocks of block_size tokens and a
 * block table maps each sequence's logical blocks to physical ones).
 *   q                   [B, num_heads, 1, D] or [B, 1, num_heads, D], device bf16
 *   k_cache, v_cache    device bf16 block pools in kv_layout:
 *                       FA_LAYOUT_PA_BBND [num_blocks, block_size, KV_N, D] or
 *                       FA_LAYOUT_PA_BNBD [num_blocks, KV_N, block_size, D]
 *   block_table         device int32 [B, max_blocks_per_seq]; token r of
 *                       sequence b is row r % block_size of block
 *                       block_table[b * max_blocks_per_seq + r / block_size].
 *                       Entries past a sequence's last block are never read;
 *                       an entry outside [0, num_blocks) reads zeros.
 *   block_size          in [16, 1024], a multiple of 16
 *   key_mask            NULL or device uint8 [B, max_blocks_per_seq * block_size]
 *   actual_seq_lengths  HOST int64 [B], required, each in
 *                       [0, max_blocks_per_seq * block_size]
 *   the rest as for fa_decode; the workspace is
 *   fa_decode_workspace_size(B, max_blocks_per_seq * block_size, ...).
 * Errors: a bad kv_layout or block_size, or negative counts ->
 * FA_ERR_PARAM_INVALID; block_table NULL with B > 0 -> FA_ERR_NULLPTR;
 * otherwise those of fa_decode. */
fa_status fa_decode_paged(const void* q, const void* k_cache, const void* v_cache, int kv_layout,
                          const int32_t* block_table, int64_t max_blocks_per_seq,
                          int64_t num_blocks, int64_t block_size, const uint8_t* key_mask,
                          const int64_t* actual_seq_lengths, int64_t B, int64_t num_heads,
                          int64_t num_kv_heads, int64_t D, float scale, int num_splits, void* out,
                          float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* The decode split plan for these arguments (pure host computation, no
 * CUDA call). Every (batch, KV head, group of query heads handled together)
 * is a unit of L_b key rows; the units are laid end to end and cut into
 * equal contiguous shares, one per CTA (the load-balancing idea of the
 * FlashAttn guide §4, SectionStreamK; splitting S2 when B*N2 is small,
 * aclnnIncreFlashAttention guide §8.2). A unit crossed by share boundaries
 * is computed in pieces that are merged by their log-sum-exp.
 * With num_splits = 0 the shares are equal in cost: a row costs 1 and the
 * start of every unit after the first costs c * 128 / D rows more, the work
 * of the piece end it brings, with c = 192 when the non-empty units outnumber
 * num_sms (so that a share holds several unit starts), c = 384 when they do
 * not but a CTA handles four or more query heads (the most costly piece
 * end), else 0; a share holding unit starts then takes fewer rows. Row x of
 * unit k costs x + that cost * k.
 *   chunk_rows  cost of a share: with num_splits = 0, the total cost divided
 *               by num_sms (at least 224); with n > 0, ceil(S_kv_max / n)
 *               rounded up to a multiple of 64, and a row costs 1
 *   num_chunks  number of shares (CTAs)
 *   max_chunks  largest number of pieces of one unit
 * num_sms is the SM count the plan is made for (fa_decode passes the
 * device's). */
fa_status fa_decode_plan(int64_t B, int64_t S_kv_max, int64_t num_heads, int64_t num_kv_heads,
                         int64_t D, const int64_t* actual_seq_lengths, int num_sms,
                         int num_splits, int64_t* chunk_rows, int64_t* num_chunks,
                         int64_t* max_chunks);

/* ------------------------------------------------------- decode, no alloc
 * fa_decode for callers that cannot allocate device memory: for example a
 * runtime that must not call cudaMalloc (allocation is forbidden while a
 * stream is being captured into a CUDA graph), a plugin that may not touch
 * its host framework's memory pool, or an embedded loader with no device
 * allocator at all. It takes the same arguments as fa_decode minus the
 * workspace; its scratch is one array of FA_NOALLOC_SCRATCH_BYTES in device
 * global memory that the library owns: every GPU that loads the library
 * holds that array until the process exits. This entry point has no
 * counterpart on the pages; it is a packaging variant of fa_decode.
 *   - Limits: the part of the array this call's split plan uses (the plan
 *     fa_decode would make for these lengths on this device; its partial
 *     results take 4 * B * num_heads * (D + 1) bytes per piece slot, none
 *     when no sequence is cut) must fit in FA_NOALLOC_SCRATCH_BYTES, else
 *     FA_ERR_WORKSPACE_TOO_SMALL; B must be at most 1024, else
 *     FA_ERR_PARAM_INVALID. Nothing is enqueued then. (The long-context
 *     shape B = 1, 32 heads, D = 128, 131072 keys needs well under 1 MiB.)
 *   - Every argument is checked before any CUDA call. Each call then looks
 *     up the array's device address on the current device; the first call
 *     on a device may load the library's device code there (which creates
 *     the array), so make that first call before any stream capture.
 *   - All calls on a device share the one array: calls whose GPU work
 *     overlaps (other streams, other threads) race and must be serialised by
 *     the caller. Each call clears the part of the array it needs cleared.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call,
 *     and the library's own code makes no host heap allocation on this path
 *     (the CUDA runtime and driver may allocate internally on first use).
 *   - A device-side timeout (FA_ERR_DEVICE_TIMEOUT) is recorded in the
 *     array's status word: read it with fa_decode_noalloc_status. */
#define FA_NOALLOC_SCRATCH_BYTES (8u << 20)

fa_status fa_decode_noalloc(const void* q, const void* k, const void* v, const uint8_t* key_mask,
                            const int64_t* actual_seq_lengths, int64_t B, int64_t S_kv_max,
                            int64_t num_heads, int64_t num_kv_heads, int64_t D, float scale,
                            int layout, int num_splits, void* out, float* lse, void* stream);

/* Status of the fa_decode_noalloc calls on the current device, as
 * fa_workspace_status gives it for a workspace: synchronises `stream`, then
 * reads and clears the status word of the library-owned array. Returns FA_OK,
 * FA_ERR_DEVICE_TIMEOUT (a bounded wait in a kernel expired) or
 * FA_ERR_RUNTIME. No counterpart on the pages (see fa_decode_noalloc). */
fa_status fa_decode_noalloc_status(void* stream);

/* ------------------------------------------------------------ diagnostics
 * Synchronises `stream`, then reads and clears the device status word at
 * the start of a workspace used by fa_forward / fa_decode. Returns FA_OK,
 * FA_ERR_DEVICE_TIMEOUT (a bounded wait in a kernel expired),
 * FA_ERR_DEVICE_CHECK (debug builds: an index check failed) or
 * FA_ERR_RUNTIME. */
fa_status fa_workspace_status(void* workspace, void* stream);

/* The bounded-wait limit (nanoseconds) of every later fa_forward* / fa_decode*
 * call made from this host thread; 0 restores the default of 2 s. Every wait
 * of the kernels on a barrier, a turn or a peer gives up after this limit:
 * the kernel records FA_ERR_DEVICE_TIMEOUT in the workspace status word (see
 * fa_workspace_status and fa_decode_noalloc_status), lets its own copies and
 * tensor-core operations in flight finish (those waits keep a limit of at
 * least 100 ms), frees what it holds and returns; its outputs are then
 * undefined. A diagnostic for failure-detection tests: a limit of a few
 * microseconds makes the first waits of a real call run out. Limits above
 * 10 s are FA_ERR_PARAM_INVALID. No counterpart on the pages. */
fa_status fa_set_wait_timeout_ns(uint64_t timeout_ns);

/* Self-test of the bounded-wait path: launches one CTA that waits on an
 * mbarrier nothing ever arrives on, with a limit of timeout_ns. The kernel
 * records FA_ERR_DEVICE_TIMEOUT's device code in the workspace's status
 * word and returns; the context stays usable. Needs >= 256 workspace bytes. */
fa_status fa_selftest_wait_timeout(void* workspace, uint64_t timeout_ns, void* stream);

/* Diagnostics for measurement. When both handles are non-NULL, every later
 * fa_forward / fa_decode call made from this host thread records `before`
 * (a cudaEvent_t) on its stream immediately before launching its main
 * kernel (the prefill kernel, or the decode stage-1 kernel) and `after`
 * immediately after it, so the pair times that kernel alone on the stream it
 * runs on. Passing NULL, NULL turns the hooks off. The events stay owned by
 * the caller. */
void fa_set_main_kernel_events(void* before, void* after);

/* Number of kernels this library has launched in this process so far. */
uint64_t fa_kernel_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
