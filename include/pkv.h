/*
 * pkv.h -- C interface of the paged GQA decode-attention library for GB300
 * (sm_103a).
 *
 * The operation (FlashQuant wiki "CUDA Kernels": flash_attention.cu "Online
 * Softmax" and "GQA (Grouped Query Attention) Support"; paged_decode.cu "Page
 * Table Addressing", "Partial Output", "Early Exit for Empty Splits";
 * split_k_reduce.cu "Algorithm"):
 *
 *   for every sequence b < B and query head h < Hq, with G = Hq / Hkv and
 *   kv = h / G (contiguous head groups), L = seq_lens[b]:
 *     k_j = k_cache[block_table[b][j / page_size], j % page_size, kv, :]
 *     v_j = v_cache[block_table[b][j / page_size], j % page_size, kv, :]
 *     s_j = scale * <q[b, h, :], k_j>                      j = 0 .. L-1
 *     out[b, h, :] = sum_j softmax(s)_j v_j                 (bf16, round to nearest even)
 *     lse[b, h]    = ln sum_j exp(s_j)                      (f32, natural log)
 *   L == 0 gives out = 0 and lse = -inf.
 *
 * The key range of every (b, kv head) is split over thread blocks (split-KV,
 * "flash-decoding"); each split keeps an online softmax in f32 and the splits
 * are merged by log-sum-exp.  The split count is a pure function of the shape
 * and the SM count (OASR "Kernel Layer", "Fused attention": the split count
 * must not depend on capture state because it changes the order the f32
 * partials are summed).
 *
 * Conventions (OASR "Kernel Layer", "Fused attention"; Atlas "CUDA Kernel
 * Engineering", "Conventions every Atlas kernel follows" and "CUDA graphs"):
 *   - every pointer is a DEVICE pointer unless marked "host";
 *   - every array is dense row-major, rightmost index contiguous;
 *   - every device pointer must be 16-byte aligned;
 *   - integers in tables are int32;
 *   - the caller owns every buffer, including the workspace: the library
 *     allocates no device memory, never synchronises inside a launch call, and
 *     its launch calls can be captured into a CUDA graph (no allocation, no
 *     synchronisation, no branch on capture state);
 *   - launch calls are asynchronous on `stream`; a bad argument returns a
 *     negative status BEFORE anything is launched; errors the device finds are
 *     recorded in a sticky status word at the start of the workspace and read
 *     back with pkv_check_status();
 *   - bf16 buffers are typed pkv_bf16 (the raw 16-bit pattern), so this header
 *     is valid C.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

typedef uint16_t pkv_bf16; /* bfloat16 bit pattern */

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = -1,         /* null pointer, non-positive size, Hq % Hkv != 0, seq bound */
    PKV_ERR_UNSUPPORTED = -2,         /* D not in {64,128,256}, page_size not a power of two in
                                         [8,256], group size Hq/Hkv > 32, B > 65535 (the
                                         sequences are a launch dimension), no sm_103a device */
    PKV_ERR_MISALIGNED = -3,          /* a device pointer is not 16-byte aligned */
    PKV_ERR_WORKSPACE_TOO_SMALL = -4, /* workspace_bytes below the size query's answer */
    PKV_ERR_CUDA = -5,                /* a CUDA runtime/driver call failed */
    PKV_ERR_BAD_PAGE_INDEX = -6,      /* device: a used block_table entry outside [0, num_pages) */
    PKV_ERR_DEVICE_TIMEOUT = -7,      /* device: a bounded wait for a copy ran out (2 s).  The
                                         block that saw it waits, bounded again, for its other
                                         copies in flight and exits; a copy that outlasts that
                                         wait too may still land in shared memory the block no
                                         longer owns.  After this status, treat the call's
                                         outputs and every later result on the same CUDA
                                         context as untrustworthy until the process restarts. */
    PKV_ERR_BAD_SEQ_LEN = -8,         /* device: seq_lens[b] < 0 or > max_pages * page_size */
    PKV_ERR_BAD_QO_INDPTR = -9        /* device: a request's query rows outside [0, total_q) or more
                                         than max_q_len of them */
} pkv_status;

/* Human-readable name of a status code (static string; never NULL). */
PKV_API const char *pkv_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
PKV_API int pkv_version(void);

/*
 * Programmatic dependent launch (PDL).  enable != 0: every later launch by this
 * library (any stream, any thread of the process) carries the
 * programmatic-stream-serialization attribute, so a kernel may begin launching
 * while the previous kernel in its stream still runs; each kernel waits for that
 * kernel's completion (griddepcontrol.wait) before reading any input, so results
 * are unchanged.  The KV append lets the following kernel launch at once; the decode
 * kernel lets it launch once its blocks have streamed their keys.  The overlap
 * hides the launch gap between the steps of a decode iteration (append, then
 * attention), also inside CUDA graphs.  Returns the previous setting (0 at load).
 */
PKV_API int pkv_set_programmatic_launch(int enable);

/*
 * Split merge through a thread-block cluster (on at load).  enable != 0: a
 * decode call whose plan has 2-8 splits and whose grid fits one wave of resident
 * blocks launches the splits of each (b, kv head) as one cluster; each split sends
 * its normalised partial output and lse into split 0's shared memory (distributed
 * shared memory, st.async), and split 0 merges them with the same log-sum-exp
 * combine, in the same split order, as the workspace merge (FlashQuant wiki
 * "CUDA Kernels", split_k_reduce.cu "Algorithm"), so the results are identical
 * bit for bit.  enable == 0: every merge goes through the workspace (the last
 * split to finish merges).  Measured on GB300, the batch workload (one wave,
 * 5-7 splits) runs 4-8% faster with it; grids of several waves never take it
 * (clusters placed whole leave slots idle there).  Process-wide, like
 * pkv_set_programmatic_launch; the plan queries report the choice in
 * pkv_plan.merge_needed.  Returns the previous setting.
 */
PKV_API int pkv_set_cluster_merge(int enable);

/*
 * Adaptive split count (off at load).  enable != 0: a decode call with the automatic split
 * count (paged_decode_attn, paged_decode_attn_fp8, paged_decode_attn_ex with num_splits = 0;
 * B <= 1024) sizes its splits on the device from the batch's actual lengths instead of the
 * block table's width (Atlas "CUDA Kernel Engineering", "The kernel inventory": adaptive split
 * count): every block reads the B lengths and takes chunks of about (sum of the lengths x Hkv /
 * block slots) keys, at least 512 KiB of cache bytes (and 256 keys), at most the planned chunk,
 * and enough that no sequence needs more than the planned split count, so the grid, the
 * workspace and the plan stay as pkv_plan_query reports them.  It pays where the table is much
 * wider than the sequences and there are few (sequence, kv head) groups (measured on GB300: a
 * 131072-key table holding four sequences of 2048 keys, 29.3 -> 23.2 us); it costs a pass over
 * the lengths in every block, the empty splits of a wide table included (16 sequences of 1000
 * keys on the same table: 25.5 -> 30.9 us), hence off by default.  Process-wide; returns the
 * previous setting.
 */
PKV_API int pkv_set_adaptive_splits(int enable);

/*
 * Tensor-core path of paged_prefill_attn and paged_prefill_attn_fp8 (D = 128 or 256,
 * scale > 0, more than 32 (token, query head) rows per (sequence, kv head) group, i.e.
 * max_q_len * Hq/Hkv > 32): the score and PV products run on tcgen05 (5th-generation tensor
 * cores, accumulators in tensor memory), one CTA per 128 or 256 rows of a group and per key
 * range (D = 256: 128 rows per CTA, 64-key tiles).  The fp8 cache takes the 128-row kernels,
 * whose converter warps dequantise each key tile (code x scale, exact) into the bf16 tile the
 * bf16 kernel reads: their results equal, bit for bit, those of the bf16 cache holding the
 * dequantised values; where a mode below names 256 rows, the fp8 cache and D = 256 take 128.
 * Key ranges
 * (num_splits = 0): when the groups' CTAs are fewer than the SMs, SMs / CTAs ranges per
 * group (one wave), else ranges of at most 8192 keys; num_splits > 0 sets the count.  A
 * group with several ranges merges them in the kernel through the workspace.  A group of
 * at most 32 rows always takes the mma.sync kernel (one block reads each key once; at
 * D = 256 a block serves at most 16 rows, so 17-32 rows take two).
 * mode:
 *   PKV_TC_OFF     such calls take the mma.sync kernel;
 *   PKV_TC_AUTO    (the setting at load) groups of 33-127 rows: 128 rows per CTA when
 *                  max_pages * page_size >= 8192 (the mma.sync kernel would read each
 *                  key once per 32 rows), else the mma.sync kernel; groups of 128 rows
 *                  or more: 256 rows per CTA when the group has that many and that grid,
 *                  B * Hkv * ceil(max_q_len * Hq/Hkv / 256) * ranges CTAs, has at least
 *                  one CTA per two SMs, else 128 rows per CTA;
 *   PKV_TC_ALWAYS  256 rows per CTA when the group has that many, else 128;
 *   PKV_TC_ROWS128 128 rows per CTA.
 * Process-wide; returns the previous mode, or PKV_ERR_INVALID_ARG for an unknown one.
 */
enum pkv_tc_mode { PKV_TC_OFF = 0, PKV_TC_AUTO = 1, PKV_TC_ALWAYS = 2, PKV_TC_ROWS128 = 3 };
PKV_API int pkv_set_prefill_tensor_cores(int mode);

/* ------------------------------------------------------------------ planning */

/*
 * What a launch will do for a shape.  Returned by pkv_plan_query; the same
 * function decides every launch, so a plan queried on the host is the plan the
 * launch uses.
 */
typedef struct {
    int num_splits;       /* S: key-range splits per (b, kv head) at full table width */
    int chunk_tokens;     /* keys per split (a multiple of stage_tokens) */
    int stage_tokens;     /* keys per pipeline stage (one TMA box row set); tensor-core kernels:
                             keys per tile (128) */
    int warps;            /* warps per thread block (tensor-core kernels: every role) */
    int ring_stages;      /* stages in flight per warp; tensor-core kernels: K stages */
    int blocks_per_sm;    /* resident thread blocks per SM the plan assumes */
    int grid_blocks;      /* thread blocks of the split kernel (S * Hkv * B) */
    int smem_bytes;       /* dynamic shared memory per block */
    int merge_needed;     /* 0: S == 1, nothing to merge; 1: the last split block of each (b, kv
                             head) to finish merges the partials through the workspace, inside
                             the same kernel launch; 2 (decode, 2 <= S <= 8): the S split blocks
                             of each (b, kv head) form a thread-block cluster and split 0 merges
                             the others' partials in its shared memory */
    size_t workspace_bytes;
    int q_tiles;          /* blocks per (b, kv head) along its query rows (1 for decode) */
    int rows_per_block;   /* (token, query head) rows one block serves: 8, 16 or 32; 128 or 256
                             when a several-rows call takes the tensor-core kernels */
} pkv_plan;

/*
 * Pure host function: the plan for a shape on a device with `num_sms` SMs.
 * num_splits > 0 forces that many splits (clamped to [1, ceil(max_pages *
 * page_size / stage_tokens)]); 0 chooses automatically.  No CUDA call.
 */
PKV_API pkv_status pkv_plan_query(int B, int Hq, int Hkv, int D, int page_size, int max_pages,
                          int num_sms, int num_splits, pkv_plan *plan /* host */);

/* KV cache element types. */
enum pkv_kv_dtype {
    PKV_KV_BF16 = 0,      /* bf16 pools (paged_decode_attn*) */
    PKV_KV_FP8_E4M3 = 1   /* e4m3 codes + f32 scales (paged_decode_attn_fp8) */
};

/*
 * pkv_plan_query for either cache type: the fp8-cache kernel has its own
 * shared-memory footprint and residency, hence its own split count and
 * workspace size.  kv_dtype other than the two above: PKV_ERR_INVALID_ARG.
 */
PKV_API pkv_status pkv_plan_query_kv(int B, int Hq, int Hkv, int D, int page_size, int max_pages, int num_sms,
                                     int num_splits, int kv_dtype, pkv_plan *plan);

/*
 * Workspace bytes that paged_decode_attn needs for this shape on `device`
 * (queries the device's SM count).  The workspace holds a 256-byte header whose
 * first int32 is the device status word, then (when the plan splits) one int32
 * completion counter per (b, kv head) and the split partials.  Allocate it
 * zeroed before its first use; the kernel returns every counter to zero, so a
 * workspace can be reused call after call without clearing it again.  Calls
 * that may overlap on the GPU must not share a workspace.
 */
PKV_API pkv_status paged_decode_attn_workspace_size(int B, int Hq, int Hkv, int D, int page_size,
                                            int max_pages, int device, size_t *bytes /* host */);

/* Same, for a forced split count (see paged_decode_attn_ex). */
PKV_API pkv_status paged_decode_attn_workspace_size_ex(int B, int Hq, int Hkv, int D, int page_size,
                                               int max_pages, int device, int num_splits,
                                               size_t *bytes /* host */);

/* Workspace bytes for either cache type (see pkv_plan_query_kv); the fp8 call needs
 * the PKV_KV_FP8_E4M3 size. */
PKV_API pkv_status paged_decode_attn_workspace_size_kv(int B, int Hq, int Hkv, int D, int page_size,
                                                       int max_pages, int device, int num_splits, int kv_dtype,
                                                       size_t *bytes);

/* ------------------------------------------------------------------ decode */

/*
 * Paged GQA decode attention (one query token per sequence).
 *
 *   q           [B, Hq, D] bf16
 *   k_cache     [num_pages, page_size, Hkv, D] bf16 (the page pool)
 *   v_cache     [num_pages, page_size, Hkv, D] bf16
 *   block_table [B, max_pages] int32: physical page of each logical page
 *   seq_lens    [B] int32: keys per sequence
 *   scale       multiplies q.k (the caller passes e.g. 1/sqrt(D))
 *   out         [B, Hq, D] bf16 (written)
 *   lse         [B, Hq] f32, natural log (written); may be NULL
 *   workspace   caller-owned device buffer of workspace_bytes bytes
 *
 * Requirements checked on the host: pointers non-NULL (lse excepted) and
 * 16-byte aligned; B >= 0 (B == 0 is a no-op); Hq, Hkv, num_pages, max_pages
 * >= 1; Hq % Hkv == 0 and Hq / Hkv <= 32; D in {64, 128, 256}; page_size a
 * power of two in [8, 256]; workspace large enough.
 *
 * Device-data preconditions (not checked on the host): 0 <= seq_lens[b] <=
 * max_pages * page_size, and block_table[b][0 .. ceil(seq_lens[b]/page_size)-1]
 * are page ids in [0, num_pages).  Entries past that are never read and may
 * hold anything; key slots past seq_lens[b] in the last page are never used
 * (they may hold NaN).  A violation is not a fault: a page id out of range is
 * skipped (its keys contribute nothing) and the status word records
 * PKV_ERR_BAD_PAGE_INDEX; a length out of range makes that sequence empty
 * (out = 0, lse = -inf) and records PKV_ERR_BAD_SEQ_LEN.  The first error
 * recorded since the last reset is kept.
 */
PKV_API pkv_status paged_decode_attn(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                             const int32_t *block_table, const int32_t *seq_lens,
                             int B, int Hq, int Hkv, int D, int page_size, int num_pages,
                             int max_pages, float scale, pkv_bf16 *out, float *lse,
                             void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Same as paged_decode_attn with a forced split count (num_splits > 0), for
 * tests and sweeps; 0 is the automatic choice.  Results for different split
 * counts differ only by f32 summation order.
 */
PKV_API pkv_status paged_decode_attn_ex(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                                const int32_t *block_table, const int32_t *seq_lens,
                                int B, int Hq, int Hkv, int D, int page_size, int num_pages,
                                int max_pages, float scale, pkv_bf16 *out, float *lse,
                                void *workspace, size_t workspace_bytes, int num_splits,
                                cudaStream_t stream);

/*
 * Decode attention for callers that cannot allocate device memory.
 *
 * Same operation, arguments and results as paged_decode_attn, without the
 * workspace: the split partials and the status word live in one fixed device
 * array inside this library (32 MiB, held on every GPU that loads the
 * library until the process exits).  It exists for callers that may not call
 * cudaMalloc at decode time -- a serving loop whose device memory pool is
 * sized and frozen at start-up, a plugin that is handed only one step's
 * tensors, a host without the runtime's allocator -- and it allocates nothing
 * itself.  The pages describe no such entry point; it is a library service.
 *
 *   device_status  device int (may be NULL): receives this call's device status
 *                  word (PKV_OK or the first device-side error) once the
 *                  kernels are done, in stream order.
 *
 * The first call on a device looks up the array's device address for that
 * device (make that call before any stream capture) and keeps it for the life
 * of the process: it is not looked up again after cudaDeviceReset or anything
 * else that tears down the device's primary context, so do not call this
 * entry point after such a reset.  A shape whose plan
 * needs more than 32 MiB of partials returns PKV_ERR_WORKSPACE_TOO_SMALL
 * before anything runs; use paged_decode_attn with a workspace for those.
 * Every call first clears the status word and the split-completion
 * counters.  All calls on a device share the array: calls that may overlap
 * on the GPU (other streams, other host threads) race on it and must be
 * ordered by the caller.  A call rejected on the host (a bad argument, a
 * misaligned pointer, too large a plan) touches neither the GPU nor the array.
 */
PKV_API pkv_status paged_decode_attn_static_scratch(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                                                    const pkv_bf16 *v_cache, const int32_t *block_table,
                                                    const int32_t *seq_lens, int B, int Hq, int Hkv, int D,
                                                    int page_size, int num_pages, int max_pages, float scale,
                                                    pkv_bf16 *out, float *lse, int *device_status,
                                                    cudaStream_t stream);

/* ------------------------------------------------------------------ append */

/*
 * Paged KV append: the per-token cache write that precedes a decode step
 * (Atlas "CUDA Kernel Engineering", "The kernel inventory": KV append, a
 * per-token K/V write into the paged cache).  For every sequence b and kv head
 * g, copies k_new[b, g, :] and v_new[b, g, :] into
 *   k_cache / v_cache[block_table[b][pos / page_size], pos % page_size, g, :]
 * with pos = positions[b] (normally the sequence's length before the step; the
 * caller then passes seq_lens + 1 to the decode call).  One launch, K and V
 * together, asynchronous on `stream`.
 *
 *   k_new, v_new  [B, Hkv, D] bf16
 *   block_table   [B, max_pages] int32 (the same table the decode call reads)
 *   positions     [B] int32; a negative position skips that sequence
 *   k_cache, v_cache [num_pages, page_size, Hkv, D] bf16 (written in place)
 *   status        device int32 or NULL; the first device-side error is
 *                 recorded there when it holds 0 -- the decode workspace
 *                 pointer can be passed (its first int32 is the status word)
 * Host checks as for paged_decode_attn (D in {64,128,256}, power-of-two
 * page_size in [8,256], 16-byte alignment).  Device: a position >=
 * max_pages * page_size records PKV_ERR_BAD_SEQ_LEN, a page id outside
 * [0, num_pages) records PKV_ERR_BAD_PAGE_INDEX; that sequence is not written.
 * Every other byte of the pools is left untouched.
 */
PKV_API pkv_status paged_kv_append(const pkv_bf16 *k_new, const pkv_bf16 *v_new, const int32_t *block_table,
                                   const int32_t *positions, int B, int Hkv, int D, int page_size, int num_pages,
                                   int max_pages, pkv_bf16 *k_cache, pkv_bf16 *v_cache, int *status,
                                   cudaStream_t stream);

/* ------------------------------------------------------------------ fp8 cache */

/*
 * FP8 KV cache (OASR "Kernel Layer", "FP8 KV variants"): the pools hold float8
 * e4m3 codes ("fn" variant: sign, 4 exponent bits with bias 7, 3 mantissa bits,
 * no infinities, S.1111.111 = NaN, largest finite 448) with one f32 scale per
 * (token, kv head).  The key (value) element used for slot t of page p, kv head
 * g, dim d is
 *     code(k_cache[p, t, g, d]) * k_scale[p, g, t]
 * The kernel decodes the codes exactly into f16 and runs the f16 tensor-core
 * mma with f32 accumulation; the key scale multiplies the score, the value scale
 * the probability, so any positive finite scale is honoured (the power-of-two
 * scales paged_kv_append_fp8 writes make code * scale exactly representable in
 * bf16 as well).  The plan (split count, chunk, workspace size) is
 * pkv_plan_query_kv's with PKV_KV_FP8_E4M3.  Results match the bf16 kernel run
 * on a bf16 cache holding code * scale up to the rounding of the probabilities
 * and the f32 summation order.
 *
 *   k_cache, v_cache  [num_pages, page_size, Hkv, D] uint8 e4m3 codes
 *   k_scale, v_scale  [num_pages, Hkv, page_size] f32 (head-major within a page,
 *                     so one head's scales for a page are contiguous), 16-byte
 *                     aligned
 * Every other argument, the workspace (size from
 * paged_decode_attn_workspace_size_kv with PKV_KV_FP8_E4M3 and the same
 * num_splits), the status word and the error behaviour are those of
 * paged_decode_attn_ex.  NaN codes
 * or scales in slots past seq_lens[b] are never used.
 */
PKV_API pkv_status paged_decode_attn_fp8(const pkv_bf16 *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                         const float *k_scale, const float *v_scale, const int32_t *block_table,
                                         const int32_t *seq_lens, int B, int Hq, int Hkv, int D, int page_size,
                                         int num_pages, int max_pages, float scale, pkv_bf16 *out, float *lse,
                                         void *workspace, size_t workspace_bytes, int num_splits,
                                         cudaStream_t stream);

/*
 * Quantise-and-append into an fp8 cache: paged_kv_append's write, quantising
 * each new (sequence, kv head) row of K and of V on the way, K and V in one
 * launch (OASR "Kernel Layer", "FP8 KV variants": one quantise-and-scatter
 * launch writes the cache).  A row x of D values gets
 *     scale = 2^k, k the smallest integer in [-64, 64] with max_d |x_d| <= 448 * 2^k
 *     code_d = e4m3(x_d / scale), round to nearest even, saturating at +-448
 * (NaN values are left out of the maximum and give a NaN code).  The codes go to
 * k_cache/v_cache[page, slot, g, :] and the scale to k_scale/v_scale[page, g,
 * slot], with page and slot from positions[b] as in paged_kv_append.  Every
 * other argument and the error behaviour are those of paged_kv_append; the
 * scale tensors are [num_pages, Hkv, page_size] f32, 16-byte aligned.  Calling
 * it with B = num_pages * page_size rows, a one-page table per row and
 * positions = slot quantises a whole pool in one launch.
 */
PKV_API pkv_status paged_kv_append_fp8(const pkv_bf16 *k_new, const pkv_bf16 *v_new, const int32_t *block_table,
                                       const int32_t *positions, int B, int Hkv, int D, int page_size,
                                       int num_pages, int max_pages, uint8_t *k_cache, uint8_t *v_cache,
                                       float *k_scale, float *v_scale, int *status, cudaStream_t stream);

/* ------------------------------------------------------------------ several query rows */

/*
 * Several query rows per sequence: multi-token decode (speculative or
 * multi-token prediction steps) and chunked paged prefill (AstrAI "CUDA Kernels",
 * "Q Scheduling and KV Addressing": a packed [total_q, Hq, D] query tensor,
 * qo_indptr, paged KV, the query heads of one kv-head group sharing each K/V
 * tile).  Request b owns query rows qo_indptr[b] .. qo_indptr[b+1]-1 (n_b rows)
 * and seq_lens[b] = L_b keys, the new tokens' keys included (append them first).
 * The new tokens are the request's last n_b positions: with causal = 1, row i
 * (0-based within the request) attends to keys j <= L_b - n_b + i; with
 * causal = 0 to all L_b keys.  A row that sees no key gives out = 0, lse = -inf.
 *
 *   q, out      [total_q, Hq, D] bf16;  lse [total_q, Hq] f32 (may be NULL)
 *   qo_indptr   [B+1] int32 device, qo_indptr[0] = 0, non-decreasing,
 *               qo_indptr[B] = total_q, every n_b <= max_q_len
 *   max_q_len   the most rows a request has (sizes the grid: a block serves up to
 *               32 (token, query head) rows of one kv-head group; see
 *               pkv_plan_query_prefill's q_tiles)
 * Everything else as paged_decode_attn_ex (the fp8 form as paged_decode_attn_fp8).
 * Workspace: paged_prefill_attn_workspace_size.  A request whose row range breaks
 * the contract is skipped (nothing read or written for it) and
 * PKV_ERR_BAD_QO_INDPTR is recorded.  Decode is the case qo_indptr[b] = b,
 * max_q_len = 1.  Groups of at most 32 rows run on the mma.sync kernel, which reads
 * the K/V stream once per query tile of up to 32 rows (16 at D = 256); larger groups may run on the
 * tensor-core kernels (pkv_set_prefill_tensor_cores), which read it once per 128 or
 * 256 rows.
 */
PKV_API pkv_status paged_prefill_attn(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                                      const int32_t *qo_indptr, const int32_t *block_table,
                                      const int32_t *seq_lens, int B, int Hq, int Hkv, int D, int page_size,
                                      int num_pages, int max_pages, int total_q, int max_q_len, int causal,
                                      float scale, pkv_bf16 *out, float *lse, void *workspace,
                                      size_t workspace_bytes, int num_splits, cudaStream_t stream);

PKV_API pkv_status paged_prefill_attn_fp8(const pkv_bf16 *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                          const float *k_scale, const float *v_scale, const int32_t *qo_indptr,
                                          const int32_t *block_table, const int32_t *seq_lens, int B, int Hq,
                                          int Hkv, int D, int page_size, int num_pages, int max_pages,
                                          int total_q, int max_q_len, int causal, float scale, pkv_bf16 *out,
                                          float *lse, void *workspace, size_t workspace_bytes, int num_splits,
                                          cudaStream_t stream);

/* The plan of a several-rows call (kv_dtype as pkv_plan_query_kv), under the tensor-core
 * routing set when it is queried and for a positive scale (a call with scale <= 0 takes the
 * mma.sync kernel): when the routing takes the tensor cores, the launch fields are the
 * tensor-core kernel's (rows_per_block 128 or 256).  workspace_bytes covers the mma.sync
 * kernel and every tensor-core kernel the call could take under any routing. */
PKV_API pkv_status pkv_plan_query_prefill(int B, int Hq, int Hkv, int D, int page_size, int max_pages, int total_q,
                                          int max_q_len, int num_sms, int num_splits, int kv_dtype,
                                          pkv_plan *plan);

/* Workspace bytes of a several-rows call on `device`. */
PKV_API pkv_status paged_prefill_attn_workspace_size(int B, int Hq, int Hkv, int D, int page_size, int max_pages,
                                                     int total_q, int max_q_len, int device, int num_splits,
                                                     int kv_dtype, size_t *bytes);

/* ------------------------------------------------------------------ merge */

/*
 * Log-sum-exp merge of S per-split partial results (FlashQuant wiki "CUDA
 * Kernels", split_k_reduce.cu "Algorithm" and "Numerical Stability"), in the
 * self-contained form: each split passes its softmax-normalised output and
 * its natural-log LSE.
 *
 *   partial_out [S, B, Hq, D] f32   split s's output over its own keys
 *   partial_lse [S, B, Hq] f32      split s's LSE; -inf marks an empty split
 *   out         [B, Hq, D] bf16     sum_s w_s o_s / sum_s w_s,  w_s = exp(lse_s - max_s lse_s)
 *   lse         [B, Hq] f32         max + ln sum_s w_s; may be NULL
 * Every split empty gives out = 0 and lse = -inf.  S >= 1, D in {64,128,256}.
 * This is also the combine step a caller would run after gathering partials
 * produced elsewhere (for example by another device holding part of the keys).
 */
PKV_API pkv_status split_kv_merge(const float *partial_out, const float *partial_lse, int S, int B,
                          int Hq, int D, pkv_bf16 *out, float *lse, cudaStream_t stream);

/* ------------------------------------------------------------------ status */

/*
 * Synchronises `stream`, then copies the workspace's device status word into
 * *device_status (host): PKV_OK or the first device-side error recorded since
 * the last reset.  Returns PKV_ERR_CUDA if the synchronisation or copy fails.
 */
PKV_API pkv_status pkv_check_status(const void *workspace, cudaStream_t stream, int *device_status /* host */);

/* Zeroes the workspace's status word, asynchronously on `stream`. */
PKV_API pkv_status pkv_reset_status(void *workspace, cudaStream_t stream);

/*
 * Diagnostic: launches one block that waits, with the same bounded wait the
 * decode kernel uses, on a barrier that nothing ever completes, for at most
 * `timeout_us` microseconds, then records PKV_ERR_DEVICE_TIMEOUT in the
 * workspace status word and returns.  Lets a test check that a stalled copy
 * ends in a status code rather than a hang.
 */
PKV_API pkv_status pkv_selftest_wait_timeout(void *workspace, unsigned timeout_us, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
