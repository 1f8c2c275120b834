// api.cu -- the C-ABI entry points declared in include/pkv.h.
//
// Host side of the library: argument checks (before any launch), the plan,
// the TMA tensor-map cache, and the kernel launches.  Launch calls never
// allocate device memory and never synchronise.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <algorithm>
#include <atomic>

#include "append_kernel.cuh"
#include "decode_launch.cuh"
#include "launch_util.h"
#include "prefill_tc2_kernel.cuh"
#include "prefill_tc256_kernel.cuh"
#include "prefill_tc_kernel.cuh"
#include "merge_kernel.cuh"
#include "pkv.h"
#include "plan.h"
#include "tc_plan.h"

namespace pkv {

std::atomic<int> g_pdl{0};
bool pdl_enabled() { return g_pdl.load(std::memory_order_relaxed) != 0; }
std::atomic<int> g_prefill_tc{PKV_TC_AUTO};
std::atomic<int> g_cluster_merge{1};
bool cluster_merge_enabled() { return g_cluster_merge.load(std::memory_order_relaxed) != 0; }
std::atomic<int> g_adaptive_splits{0};
bool adaptive_splits_enabled() { return g_adaptive_splits.load(std::memory_order_relaxed) != 0; }

namespace {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s: far above any healthy copy
// Several-rows routing: a group of at most kMqBlockRows (token, head) rows fits one block of
// the mma.sync kernel, which then reads each key once; larger groups may take the tensor
// cores, groups below 128 rows only when the block table spans kTcShortGroupKeys keys or more
// (measured on GB300: 64-row groups on 32K- and 128K-key tables 1.5-1.8x faster there, on a
// 4K-key table 12% slower).
constexpr int kMqBlockRows = 32;
constexpr long kTcShortGroupKeys = 8192;
// Largest batch whose decode blocks rank the sequence lengths themselves (longest first).
constexpr int kLongestFirstMaxB = 128;
// Largest batch whose decode sizes its splits from the actual lengths on the device (every
// block reads the B lengths: 8 loads a thread at most).
constexpr int kAdaptMaxB = 1024;
constexpr long kAdaptMinSplitBytes = 512l << 10;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int log2_exact(int x)
{
    int r = 0;
    while ((1 << r) < x) ++r;
    return r;
}

// ---------------------------------------------------------------- tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

struct MapKey {
    const void *ptr;
    int num_pages, P, Hkv, D, box_t, device, rank;  // rank 8: the fp8 (byte) view
    bool operator==(const MapKey &o) const
    {
        return ptr == o.ptr && num_pages == o.num_pages && P == o.P && Hkv == o.Hkv && D == o.D &&
               box_t == o.box_t && device == o.device && rank == o.rank;
    }
};

struct MapCache {
    static constexpr int N = 64;
    MapKey keys[N];
    CUtensorMap maps[N];
    bool used[N] = {};
    int next = 0;
    std::mutex mu;
};

MapCache &map_cache()
{
    static MapCache c;
    return c;
}

// Tensor maps over the page pool (bf16, 128-byte swizzle), cached per (pointer,
// shape, device, rank):
//   rank 4: dims (64 dims, num_pages*P rows, D/64 column blocks, Hkv heads) with
//           strides (row: Hkv*D*2 B, column block: 128 B, head: D*2 B); one box
//           (64, box_t, D/64, 1) lands a page slice of one head as [D/64][box_t][64];
//   rank 3: dims (D, Hkv, num_pages*P rows), box (64, 1, box_t): one box per
//           64-column block (the fallback when the driver refuses the rank-4 view);
//   rank 8 (the fp8 pool, bytes): the rank-4 view with INNER = min(D, 128) bytes
//           per column block: dims (INNER, num_pages*P rows, D/INNER, Hkv), strides
//           (Hkv*D B, INNER B, D B), box (INNER, box_t, D/INNER, 1), 128-byte
//           swizzle (64-byte for D = 64): a page slice of one head lands as
//           [D/INNER][box_t][INNER] codes.
pkv_status get_pool_map(const void *pool, int num_pages, int P, int Hkv, int D, int box_t, int device, int rank,
                        CUtensorMap *out)
{
    MapKey key{pool, num_pages, P, Hkv, D, box_t, device, rank};
    MapCache &c = map_cache();
    std::lock_guard<std::mutex> lock(c.mu);
    for (int i = 0; i < MapCache::N; ++i)
        if (c.used[i] && c.keys[i] == key) {
            *out = c.maps[i];
            return PKV_OK;
        }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return PKV_ERR_CUDA;
    CUtensorMap m;
    CUresult r;
    if (rank == 8) {
        const int inner = D < 128 ? D : 128;
        const cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)num_pages * (cuuint64_t)P,
                                    (cuuint64_t)(D / inner), (cuuint64_t)Hkv};
        const cuuint64_t strides[3] = {(cuuint64_t)Hkv * D, (cuuint64_t)inner, (cuuint64_t)D};
        const cuuint32_t box[4] = {(cuuint32_t)inner, (cuuint32_t)box_t, (cuuint32_t)(D / inner), 1u};
        const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
        r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(pool), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, inner == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else if (rank == 4) {
        const cuuint64_t dims[4] = {64u, (cuuint64_t)num_pages * (cuuint64_t)P, (cuuint64_t)(D / 64),
                                    (cuuint64_t)Hkv};
        const cuuint64_t strides[3] = {(cuuint64_t)Hkv * D * 2, 128u, (cuuint64_t)D * 2};
        const cuuint32_t box[4] = {64u, (cuuint32_t)box_t, (cuuint32_t)(D / 64), 1u};
        const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
        r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(pool), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)num_pages * (cuuint64_t)P};
        const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2};
        const cuuint32_t box[3] = {64u, 1u, (cuuint32_t)box_t};
        const cuuint32_t estr[3] = {1u, 1u, 1u};
        r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(pool), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return PKV_ERR_CUDA;
    const int slot = c.next;
    c.next = (c.next + 1) % MapCache::N;
    c.keys[slot] = key;
    c.maps[slot] = m;
    c.used[slot] = true;
    *out = m;
    return PKV_OK;
}

// ---------------------------------------------------------------- device facts

pkv_status current_device_sms(int *device, int *sms)
{
    if (cudaGetDevice(device) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *device) != cudaSuccess) return PKV_ERR_CUDA;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *device);
    if (major != 10 || minor != 3) return PKV_ERR_UNSUPPORTED;  // built for sm_103a only
    return PKV_OK;
}

// ---------------------------------------------------------------- launches

// Bounded-wait self-test: waits on a barrier nothing completes.
__global__ void wait_timeout_selftest_kernel(int *status, unsigned long long limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(smem_addr(&bar), 1);
    fence_barrier_init();
    if (!mbar_wait_bounded(smem_addr(&bar), 0, limit_ns)) record_status(status, PKV_ERR_DEVICE_TIMEOUT);
}


pkv_status launch_merge(int D, const MergeParams &mp, cudaStream_t stream)
{
    const int rows = mp.B * mp.Hq;
    dim3 grid((rows + kMergeWarps - 1) / kMergeWarps), block(kMergeWarps * 32);
    switch (D) {
        case 64: return launch_kernel(merge_kernel<64>, grid, block, 0, stream, mp) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
        case 128: return launch_kernel(merge_kernel<128>, grid, block, 0, stream, mp) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
        case 256: return launch_kernel(merge_kernel<256>, grid, block, 0, stream, mp) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
        default: return PKV_ERR_UNSUPPORTED;
    }
}

// The fp8 cache's scale tensors (on == false: a bf16 cache).
struct Fp8Scales {
    bool on = false;
    const float *k_scale = nullptr, *v_scale = nullptr;
};

// Several query rows per sequence (qo_indptr == nullptr: decode, one row each).
struct MultiRows {
    const int32_t *qo_indptr = nullptr;
    int total_q = 0, max_q_len = 0, causal = 0;
};

// Several rows per sequence with more than 32 rows per (sequence, kv head) group (the routing
// of tensor_core_rows), D = 128 or 256, scale > 0: a tensor-core kernel, one
// CTA per cta_rows (128: prefill_tc_kernel.cuh, bf16 or fp8 cache, or prefill_tc256_kernel.cuh
// at D = 256; 256: prefill_tc2_kernel.cuh, bf16) rows and key split (tc_split_plan).
// With one split the workspace holds only the status word; with several, also the split
// counters and the per-split partial outputs and lse that the last split merges.
pkv_status prefill_tc(const pkv_bf16 *q, const void *k_cache, const void *v_cache, const Fp8Scales &fp8,
                      const int32_t *block_table, const int32_t *seq_lens, int B, int Hq, int Hkv, int page_size,
                      int num_pages, int max_pages, float scale, pkv_bf16 *out, float *lse, void *workspace,
                      size_t workspace_bytes, int num_splits, const MultiRows &mr, int device, int sms,
                      cudaStream_t stream, int cta_rows, int D)
{
    if (fp8.on && cta_rows != kTcRows) return PKV_ERR_UNSUPPORTED;  // the fp8 cache has 128-row kernels only
    if (D != 128 && (D != 256 || cta_rows != kTcRows)) return PKV_ERR_UNSUPPORTED;
    const bool two = cta_rows == kTc2Rows;
    const int variant = D == 256 ? (fp8.on ? 4 : 3) : fp8.on ? 2 : two ? 1 : 0;
    const TcSplit sp =
        tc_split_plan(B, Hq, Hkv, page_size, max_pages, mr.total_q, mr.max_q_len, num_splits, cta_rows, sms, D);
    if (workspace_bytes < sp.ws.total) return PKV_ERR_WORKSPACE_TOO_SMALL;
    const int tile_keys = tc_tile_keys(D);
    const int box_t = page_size < tile_keys ? page_size : tile_keys;
    CUtensorMap mk, mv;
    // bf16: K per 64-dim half (rank 3), V one copy per page box (rank 4); fp8: the codes of a
    // page box in one copy each (the byte view)
    pkv_status st = get_pool_map(k_cache, num_pages, page_size, Hkv, D, box_t, device, fp8.on ? 8 : 3, &mk);
    if (st != PKV_OK) return st;
    st = get_pool_map(v_cache, num_pages, page_size, Hkv, D, box_t, device, fp8.on ? 8 : 4, &mv);
    if (st != PKV_OK) return st;
    const int G = Hq / Hkv;
    const long q_tiles = sp.q_tiles;
    if ((long)Hkv * q_tiles >= (1l << 31) || B > 65535) return PKV_ERR_UNSUPPORTED;
    static bool attr_set[5][64] = {};
    static std::mutex mu;
    if (device < 0 || device >= 64) return PKV_ERR_UNSUPPORTED;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[variant][device]) {
            const cudaError_t e =
                variant == 4 ? cudaFuncSetAttribute(prefill_tc256_kernel<true>,
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize, T2568Smem::dynamic)
                : variant == 3 ? cudaFuncSetAttribute(prefill_tc256_kernel<false>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize, T256Smem::dynamic)
                : variant == 1 ? cudaFuncSetAttribute(prefill_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                      Tc2Smem::dynamic)
                : variant == 2 ? cudaFuncSetAttribute(prefill_tc_kernel<true>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize, Tc8Smem::dynamic)
                               : cudaFuncSetAttribute(prefill_tc_kernel<false>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize, TcSmem::dynamic);
            if (e != cudaSuccess) return PKV_ERR_CUDA;
            attr_set[variant][device] = true;
        }
    }
    PrefillTcParams p;
    p.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    p.qo_indptr = mr.qo_indptr;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.lse = lse;
    p.status = static_cast<int *>(workspace);
    p.k_scale = fp8.k_scale;
    p.v_scale = fp8.v_scale;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.counters = reinterpret_cast<int *>(ws + sp.ws.counters);
    p.part_lse = reinterpret_cast<float *>(ws + sp.ws.part_lse);
    p.part_out = reinterpret_cast<float *>(ws + sp.ws.part_out);
    p.total_rows = (size_t)mr.total_q * Hq;
    p.chunk_tiles = sp.chunk_tiles;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = G;
    p.P = page_size;
    p.log2P = log2_exact(page_size);
    p.num_pages = num_pages;
    p.max_pages = max_pages;
    p.total_q = mr.total_q;
    p.max_q_len = mr.max_q_len;
    p.causal = mr.causal;
    p.q_tiles = (int)q_tiles;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634074);
    p.wait_limit_ns = kWaitLimitNs;
    const dim3 grid((unsigned)(Hkv * q_tiles), (unsigned)sp.splits, (unsigned)B);
    const cudaError_t e =
        variant == 4 ? launch_kernel(prefill_tc256_kernel<true>, grid, dim3(kT2568Threads), (size_t)T2568Smem::dynamic,
                                     stream, mk, mv, p)
        : variant == 3 ? launch_kernel(prefill_tc256_kernel<false>, grid, dim3(kT256Threads),
                                       (size_t)T256Smem::dynamic, stream, mk, mv, p)
        : variant == 1
            ? launch_kernel(prefill_tc2_kernel, grid, dim3(kTc2Threads), (size_t)Tc2Smem::dynamic, stream, mk, mv, p)
        : variant == 2 ? launch_kernel(prefill_tc_kernel<true>, grid, dim3(kTc8Threads), (size_t)Tc8Smem::dynamic,
                                       stream, mk, mv, p)
                       : launch_kernel(prefill_tc_kernel<false>, grid, dim3(kTcThreads), (size_t)TcSmem::dynamic,
                                       stream, mk, mv, p);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// Rows per CTA of the tensor-core kernel a several-rows call takes (0: the mma.sync kernel),
// for a call the tensor-core kernels apply to (more than kMqBlockRows rows per group).
// Auto: groups of fewer than 128 rows take the 128-row kernel when the block table spans at
// least kTcShortGroupKeys keys (the mma.sync kernel would read every key once per 32-row
// block), else the mma.sync kernel; larger groups take 256 rows when the group has them and
// that grid (with its key splits) has at least half a CTA per SM, else 128 rows; both
// tensor-core kernels split long groups' keys.
int tensor_core_rows(int mode, int B, int Hq, int Hkv, int page_size, int max_pages, const MultiRows &mr,
                     int num_splits, long group_rows, int sms)
{
    switch (mode) {
    case PKV_TC_ALWAYS: return group_rows >= kTc2Rows ? kTc2Rows : kTcRows;
    case PKV_TC_ROWS128: return kTcRows;
    case PKV_TC_AUTO: {
        if (group_rows < kTcRows) return (long)max_pages * page_size >= kTcShortGroupKeys ? kTcRows : 0;
        if (group_rows < kTc2Rows) return kTcRows;
        const TcSplit sp =
            tc_split_plan(B, Hq, Hkv, page_size, max_pages, mr.total_q, mr.max_q_len, num_splits, kTc2Rows, sms);
        return 2l * B * Hkv * sp.q_tiles * sp.splits >= sms ? kTc2Rows : kTcRows;
    }
    default: return 0;
    }
}

// The host checks of a decode call that need neither the device nor a plan, in the order the
// entry points report them: sizes and scale, the shape, then (B > 0) null pointers, 16-byte
// alignment and the pool's key count.  own_scratch: the call's workspace is the library's own
// array, so `workspace` is not checked.  Returns PKV_OK with *nothing_to_do set for B == 0.
pkv_status check_decode_args(const pkv_bf16 *q, const void *k_cache, const void *v_cache, const Fp8Scales &fp8,
                             const int32_t *block_table, const int32_t *seq_lens, int B, int Hq, int Hkv, int D,
                             int page_size, int num_pages, int max_pages, float scale, const pkv_bf16 *out,
                             const float *lse, const void *workspace, bool own_scratch, int num_splits,
                             bool *nothing_to_do)
{
    *nothing_to_do = false;
    if (num_pages <= 0 || num_splits < 0 || !std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
    const pkv_status shape_ok = validate_shape(B, Hq, Hkv, D, page_size, max_pages);
    if (shape_ok != PKV_OK) return shape_ok;
    if (B == 0) {
        *nothing_to_do = true;
        return PKV_OK;
    }
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out || (!own_scratch && !workspace))
        return PKV_ERR_INVALID_ARG;
    if (fp8.on && (!fp8.k_scale || !fp8.v_scale)) return PKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(block_table) ||
        !aligned16(seq_lens) || !aligned16(out) || (lse && !aligned16(lse)) || (!own_scratch && !aligned16(workspace)))
        return PKV_ERR_MISALIGNED;
    if (fp8.on && (!aligned16(fp8.k_scale) || !aligned16(fp8.v_scale))) return PKV_ERR_MISALIGNED;
    if ((long)num_pages * page_size >= (1l << 31)) return PKV_ERR_INVALID_ARG;
    return PKV_OK;
}

pkv_status decode_impl(const pkv_bf16 *q, const void *k_cache, const void *v_cache, Fp8Scales fp8,
                       const int32_t *block_table, const int32_t *seq_lens, int B, int Hq, int Hkv, int D,
                       int page_size, int num_pages, int max_pages, float scale, pkv_bf16 *out, float *lse,
                       void *workspace, size_t workspace_bytes_, int num_splits, cudaStream_t stream,
                       MultiRows mr = MultiRows{})
{
    const bool kv8 = fp8.on;
    const bool mq = mr.qo_indptr != nullptr;
    bool nothing_to_do = false;
    const pkv_status args_ok = check_decode_args(q, k_cache, v_cache, fp8, block_table, seq_lens, B, Hq, Hkv, D,
                                                 page_size, num_pages, max_pages, scale, out, lse, workspace,
                                                 false, num_splits, &nothing_to_do);
    if (args_ok != PKV_OK || nothing_to_do) return args_ok;
    if (mq && !aligned16(mr.qo_indptr)) return PKV_ERR_MISALIGNED;
    const long group_rows = mq ? (long)mr.max_q_len * (Hq / Hkv) : 0;
    const long total_rows = mq ? (long)mr.total_q * Hq : (long)B * Hq;

    int device = 0, sms = 0;
    pkv_status st = current_device_sms(&device, &sms);
    if (st != PKV_OK) return st;
    if (mq && (D == 128 || D == 256) && group_rows > kMqBlockRows && scale > 0.f) {
        int tc_rows = tensor_core_rows(g_prefill_tc.load(std::memory_order_relaxed), B, Hq, Hkv, page_size,
                                       max_pages, mr, num_splits, group_rows, sms);
        // the fp8 cache: the 128-row kernels' fp8 instantiations; D = 256: the 128-row kernel of 64-key tiles
        if ((kv8 || D == 256) && tc_rows) tc_rows = kTcRows;
        if (tc_rows)
            return prefill_tc(q, k_cache, v_cache, fp8, block_table, seq_lens, B, Hq, Hkv, page_size, num_pages,
                              max_pages, scale, out, lse, workspace, workspace_bytes_, num_splits, mr, device, sms,
                              stream, tc_rows, D);
    }
    pkv_plan plan;
    st = make_plan(B, Hq, Hkv, D, page_size, max_pages, sms, num_splits, &plan, kv8, group_rows, total_rows,
                   cluster_merge_enabled());
    if (st != PKV_OK) return st;
    if (workspace_bytes_ < plan.workspace_bytes) return PKV_ERR_WORKSPACE_TOO_SMALL;

    const int box_t = plan.stage_tokens < page_size ? plan.stage_tokens : page_size;
    CUtensorMap mk, mv;
    int box4 = 0;
    if (kv8) {
        st = get_pool_map(k_cache, num_pages, page_size, Hkv, D, box_t, device, 8, &mk);
        if (st != PKV_OK) return st;
        st = get_pool_map(v_cache, num_pages, page_size, Hkv, D, box_t, device, 8, &mv);
        if (st != PKV_OK) return st;
    } else {
        // One box per tensor per stage when a stage lies in one page (rank-4 view);
        // otherwise, or if the driver refuses that view, one box per 64 columns.
        if (plan.stage_tokens <= page_size &&
            get_pool_map(k_cache, num_pages, page_size, Hkv, D, box_t, device, 4, &mk) == PKV_OK &&
            get_pool_map(v_cache, num_pages, page_size, Hkv, D, box_t, device, 4, &mv) == PKV_OK)
            box4 = 1;
        if (!box4) {
            st = get_pool_map(k_cache, num_pages, page_size, Hkv, D, box_t, device, 3, &mk);
            if (st != PKV_OK) return st;
            st = get_pool_map(v_cache, num_pages, page_size, Hkv, D, box_t, device, 3, &mv);
            if (st != PKV_OK) return st;
        }
    }

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    DecodeParams p;
    p.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.lse = lse;
    const WorkspaceLayout wl =
        workspace_layout(plan.num_splits, (size_t)B * Hkv * plan.q_tiles, (size_t)total_rows, D);
    p.counters = reinterpret_cast<int *>(ws + wl.counters);
    p.part_lse = reinterpret_cast<float *>(ws + wl.part_lse);
    p.part_out = reinterpret_cast<float *>(ws + wl.part_out);
    p.status = reinterpret_cast<int *>(ws);
    p.k_scale = fp8.k_scale;
    p.v_scale = fp8.v_scale;
    p.qo_indptr = mr.qo_indptr;
    p.total_rows = (size_t)total_rows;
    p.q_tiles = plan.q_tiles;
    p.causal = mr.causal;
    p.total_q = mr.total_q;
    p.max_q_len = mr.max_q_len;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.P = page_size;
    p.log2P = log2_exact(page_size);
    p.num_pages = num_pages;
    p.max_pages = max_pages;
    p.chunk_tokens = plan.chunk_tokens;
    p.num_splits = plan.num_splits;
    p.box4 = box4;
    p.cluster = plan.merge_needed == 2 ? 1 : 0;
    // Grids of several waves: longest sequences first (each block ranks the B lengths itself,
    // B^2 / threads comparisons, so only for batches of at most kLongestFirstMaxB).
    p.longest_first = ((long)plan.grid_blocks > (long)sms * plan.blocks_per_sm && B > 1 &&
                       B <= kLongestFirstMaxB) ? 1 : 0;
    // Decode with the automatic split count, when switched on (pkv_set_adaptive_splits): the
    // kernel sizes the splits from the batch's actual lengths (a block reads every length, so only
    // for batches of at most kAdaptMaxB), never below kAdaptMinSplitBytes of cache bytes
    // (measured on GB300: shorter splits of short sequences cost more in start-up and merge than
    // they gain) or kMinSplitTokens keys; where the planned chunk is no larger there is nothing to
    // adapt.
    {
        const long token_bytes = kv8 ? 2l * D + 8 : 4l * D;
        const long min_tokens = std::max<long>(kMinSplitTokens, kAdaptMinSplitBytes / token_bytes);
        p.min_chunk = (int)((min_tokens + plan.stage_tokens - 1) / plan.stage_tokens * plan.stage_tokens);
    }
    const bool adapt = adaptive_splits_enabled() && !mq && num_splits == 0 && plan.num_splits > 1 &&
                       B <= kAdaptMaxB && plan.chunk_tokens > p.min_chunk;
    p.adapt_slots = adapt ? split_slots(sms, plan.blocks_per_sm, kv8) : 0;

    p.scale_log2 = (float)((double)scale * 1.4426950408889634074);
    p.wait_limit_ns = kWaitLimitNs;

    const int NT = plan.rows_per_block / 8;
    if (!mq && plan.q_tiles > 1) {
        // a decode group wider than one block (D = 256, G = 32): the several-rows variant,
        // one row per sequence (no qo_indptr), serves it as two query tiles
        p.total_q = B;
        p.max_q_len = 1;
        p.causal = 0;
    }
    if (mq || plan.q_tiles > 1)
        return kv8 ? launch_prefill_fp8(D, NT, mk, mv, p, plan, B, Hkv, device, stream)
                   : launch_prefill_bf16(D, NT, mk, mv, p, plan, B, Hkv, device, stream);
    if (p.adapt_slots > 0)
        return kv8 ? launch_decode_adapt_fp8(D, NT, mk, mv, p, plan, B, Hkv, device, stream)
                   : launch_decode_adapt_bf16(D, NT, mk, mv, p, plan, B, Hkv, device, stream);
    return kv8 ? launch_decode_fp8(D, NT, mk, mv, p, plan, B, Hkv, device, stream)
               : launch_decode_bf16(D, NT, mk, mv, p, plan, B, Hkv, device, stream);
}

// Shared checks of the two append entry points; returns PKV_OK with *skip set when B == 0.
pkv_status append_checks(const void *k_new, const void *v_new, const int32_t *block_table, const int32_t *positions,
                         int B, int Hkv, int D, int page_size, int num_pages, int max_pages, const void *k_cache,
                         const void *v_cache, const int *status, bool *skip)
{
    *skip = false;
    if (num_pages <= 0) return PKV_ERR_INVALID_ARG;
    const pkv_status shape_ok = validate_shape(B, Hkv, Hkv, D, page_size, max_pages);
    if (shape_ok != PKV_OK) return shape_ok;
    if (B == 0) {
        *skip = true;
        return PKV_OK;
    }
    if (!k_new || !v_new || !block_table || !positions || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(block_table) || !aligned16(positions) ||
        !aligned16(k_cache) || !aligned16(v_cache) || (status && (reinterpret_cast<uintptr_t>(status) & 3u)))
        return PKV_ERR_MISALIGNED;
    if ((long)num_pages * page_size >= (1l << 31) || (long)B * Hkv >= (1l << 31)) return PKV_ERR_INVALID_ARG;
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

const char *pkv_status_string(int status)
{
    switch (status) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        case PKV_ERR_MISALIGNED: return "PKV_ERR_MISALIGNED";
        case PKV_ERR_WORKSPACE_TOO_SMALL: return "PKV_ERR_WORKSPACE_TOO_SMALL";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
        case PKV_ERR_BAD_PAGE_INDEX: return "PKV_ERR_BAD_PAGE_INDEX";
        case PKV_ERR_DEVICE_TIMEOUT: return "PKV_ERR_DEVICE_TIMEOUT";
        case PKV_ERR_BAD_SEQ_LEN: return "PKV_ERR_BAD_SEQ_LEN";
        case PKV_ERR_BAD_QO_INDPTR: return "PKV_ERR_BAD_QO_INDPTR";
        default: return "PKV_UNKNOWN_STATUS";
    }
}

int pkv_version(void) { return 100; }

int pkv_set_programmatic_launch(int enable) { return g_pdl.exchange(enable ? 1 : 0); }

int pkv_set_cluster_merge(int enable) { return g_cluster_merge.exchange(enable ? 1 : 0); }

int pkv_set_adaptive_splits(int enable) { return g_adaptive_splits.exchange(enable ? 1 : 0); }

int pkv_set_prefill_tensor_cores(int mode)
{
    if (mode != PKV_TC_OFF && mode != PKV_TC_AUTO && mode != PKV_TC_ALWAYS && mode != PKV_TC_ROWS128)
        return PKV_ERR_INVALID_ARG;
    return g_prefill_tc.exchange(mode);
}

pkv_status pkv_plan_query(int B, int Hq, int Hkv, int D, int page_size, int max_pages, int num_sms, int num_splits,
                          pkv_plan *plan)
{
    return make_plan(B, Hq, Hkv, D, page_size, max_pages, num_sms, num_splits, plan, false, 0, 0,
                     cluster_merge_enabled());
}

pkv_status paged_decode_attn_workspace_size_ex(int B, int Hq, int Hkv, int D, int page_size, int max_pages,
                                               int device, int num_splits, size_t *bytes)
{
    if (!bytes) return PKV_ERR_INVALID_ARG;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return PKV_ERR_CUDA;
    pkv_plan plan;
    const pkv_status st = make_plan(B, Hq, Hkv, D, page_size, max_pages, sms, num_splits, &plan);
    if (st != PKV_OK) return st;
    *bytes = plan.workspace_bytes;
    return PKV_OK;
}

pkv_status pkv_plan_query_kv(int B, int Hq, int Hkv, int D, int page_size, int max_pages, int num_sms,
                             int num_splits, int kv_dtype, pkv_plan *plan)
{
    if (kv_dtype != PKV_KV_BF16 && kv_dtype != PKV_KV_FP8_E4M3) return PKV_ERR_INVALID_ARG;
    return make_plan(B, Hq, Hkv, D, page_size, max_pages, num_sms, num_splits, plan, kv_dtype == PKV_KV_FP8_E4M3,
                     0, 0, cluster_merge_enabled());
}

pkv_status paged_decode_attn_workspace_size_kv(int B, int Hq, int Hkv, int D, int page_size, int max_pages,
                                               int device, int num_splits, int kv_dtype, size_t *bytes)
{
    if (!bytes || (kv_dtype != PKV_KV_BF16 && kv_dtype != PKV_KV_FP8_E4M3)) return PKV_ERR_INVALID_ARG;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return PKV_ERR_CUDA;
    pkv_plan plan;
    const pkv_status st = make_plan(B, Hq, Hkv, D, page_size, max_pages, sms, num_splits, &plan,
                                    kv_dtype == PKV_KV_FP8_E4M3);
    if (st != PKV_OK) return st;
    *bytes = plan.workspace_bytes;
    return PKV_OK;
}

pkv_status paged_decode_attn_workspace_size(int B, int Hq, int Hkv, int D, int page_size, int max_pages, int device,
                                            size_t *bytes)
{
    return paged_decode_attn_workspace_size_ex(B, Hq, Hkv, D, page_size, max_pages, device, 0, bytes);
}

pkv_status paged_decode_attn(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                             const int32_t *block_table, const int32_t *seq_lens, int B, int Hq, int Hkv, int D,
                             int page_size, int num_pages, int max_pages, float scale, pkv_bf16 *out, float *lse,
                             void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    return decode_impl(q, k_cache, v_cache, Fp8Scales{}, block_table, seq_lens, B, Hq, Hkv, D, page_size,
                       num_pages, max_pages, scale, out, lse, workspace, workspace_bytes, 0, stream);
}

pkv_status paged_decode_attn_ex(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                                const int32_t *block_table, const int32_t *seq_lens, int B, int Hq, int Hkv, int D,
                                int page_size, int num_pages, int max_pages, float scale, pkv_bf16 *out, float *lse,
                                void *workspace, size_t workspace_bytes, int num_splits, cudaStream_t stream)
{
    return decode_impl(q, k_cache, v_cache, Fp8Scales{}, block_table, seq_lens, B, Hq, Hkv, D, page_size,
                       num_pages, max_pages, scale, out, lse, workspace, workspace_bytes, num_splits, stream);
}

pkv_status paged_decode_attn_fp8(const pkv_bf16 *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                 const float *k_scale, const float *v_scale, const int32_t *block_table,
                                 const int32_t *seq_lens, int B, int Hq, int Hkv, int D, int page_size,
                                 int num_pages, int max_pages, float scale, pkv_bf16 *out, float *lse,
                                 void *workspace, size_t workspace_bytes, int num_splits, cudaStream_t stream)
{
    Fp8Scales f;
    f.on = true;
    f.k_scale = k_scale;
    f.v_scale = v_scale;
    return decode_impl(q, k_cache, v_cache, f, block_table, seq_lens, B, Hq, Hkv, D, page_size, num_pages,
                       max_pages, scale, out, lse, workspace, workspace_bytes, num_splits, stream);
}

static pkv_status multi_rows(const int32_t *qo_indptr, int B, int total_q, int max_q_len, int causal,
                             MultiRows *mr)
{
    if (!qo_indptr && B > 0) return PKV_ERR_INVALID_ARG;
    if (total_q < 0 || max_q_len < 1 || (causal != 0 && causal != 1)) return PKV_ERR_INVALID_ARG;
    mr->qo_indptr = qo_indptr;
    mr->total_q = total_q;
    mr->max_q_len = max_q_len;
    mr->causal = causal;
    return PKV_OK;
}

pkv_status paged_prefill_attn(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                              const int32_t *qo_indptr, const int32_t *block_table, const int32_t *seq_lens, int B,
                              int Hq, int Hkv, int D, int page_size, int num_pages, int max_pages, int total_q,
                              int max_q_len, int causal, float scale, pkv_bf16 *out, float *lse, void *workspace,
                              size_t workspace_bytes, int num_splits, cudaStream_t stream)
{
    MultiRows mr;
    const pkv_status st = multi_rows(qo_indptr, B, total_q, max_q_len, causal, &mr);
    if (st != PKV_OK) return st;
    if (total_q == 0) return PKV_OK;
    return decode_impl(q, k_cache, v_cache, Fp8Scales{}, block_table, seq_lens, B, Hq, Hkv, D, page_size,
                       num_pages, max_pages, scale, out, lse, workspace, workspace_bytes, num_splits, stream, mr);
}

pkv_status paged_prefill_attn_fp8(const pkv_bf16 *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                  const float *k_scale, const float *v_scale, const int32_t *qo_indptr,
                                  const int32_t *block_table, const int32_t *seq_lens, int B, int Hq, int Hkv, int D,
                                  int page_size, int num_pages, int max_pages, int total_q, int max_q_len,
                                  int causal, float scale, pkv_bf16 *out, float *lse, void *workspace,
                                  size_t workspace_bytes, int num_splits, cudaStream_t stream)
{
    MultiRows mr;
    const pkv_status st = multi_rows(qo_indptr, B, total_q, max_q_len, causal, &mr);
    if (st != PKV_OK) return st;
    if (total_q == 0) return PKV_OK;
    Fp8Scales f;
    f.on = true;
    f.k_scale = k_scale;
    f.v_scale = v_scale;
    return decode_impl(q, k_cache, v_cache, f, block_table, seq_lens, B, Hq, Hkv, D, page_size, num_pages,
                       max_pages, scale, out, lse, workspace, workspace_bytes, num_splits, stream, mr);
}

pkv_status pkv_plan_query_prefill(int B, int Hq, int Hkv, int D, int page_size, int max_pages, int total_q,
                                  int max_q_len, int num_sms, int num_splits, int kv_dtype, pkv_plan *plan)
{
    if (kv_dtype != PKV_KV_BF16 && kv_dtype != PKV_KV_FP8_E4M3) return PKV_ERR_INVALID_ARG;
    if (total_q < 0 || max_q_len < 1 || Hkv <= 0) return PKV_ERR_INVALID_ARG;
    const long group_rows = (long)max_q_len * (Hq / Hkv);
    const pkv_status st = make_plan(B, Hq, Hkv, D, page_size, max_pages, num_sms, num_splits, plan,
                                    kv_dtype == PKV_KV_FP8_E4M3, group_rows, (long)total_q * Hq);
    const bool kv8 = kv_dtype == PKV_KV_FP8_E4M3;
    if (st != PKV_OK || !(D == 128 || D == 256) || group_rows <= kMqBlockRows) return st;
    // the tensor-core kernels may take the call: room for their split partials too (the fp8
    // cache and D = 256 have 128-row kernels only), whatever the routing when the call is made
    for (int rows : {kTcRows, kTc2Rows}) {
        if ((kv8 || D == 256) && rows != kTcRows) continue;
        const TcSplit sp =
            tc_split_plan(B, Hq, Hkv, page_size, max_pages, total_q, max_q_len, num_splits, rows, num_sms, D);
        plan->workspace_bytes = std::max(plan->workspace_bytes, sp.ws.total);
    }
    // the launch under the current routing (for a positive scale): a tensor-core kernel's
    // replaces the mma.sync kernel's
    MultiRows mr;
    mr.total_q = total_q;
    mr.max_q_len = max_q_len;
    int tc_rows = tensor_core_rows(g_prefill_tc.load(std::memory_order_relaxed), B, Hq, Hkv, page_size, max_pages,
                                   mr, num_splits, group_rows, num_sms);
    if ((kv8 || D == 256) && tc_rows) tc_rows = kTcRows;
    if (tc_rows) {
        const TcSplit sp =
            tc_split_plan(B, Hq, Hkv, page_size, max_pages, total_q, max_q_len, num_splits, tc_rows, num_sms, D);
        const bool d256 = D == 256;
        plan->num_splits = sp.splits;
        plan->chunk_tokens = sp.chunk_tiles * tc_tile_keys(D);
        plan->stage_tokens = tc_tile_keys(D);
        plan->warps = (d256 ? (kv8 ? kT2568Threads : kT256Threads)
                       : tc_rows == kTc2Rows ? kTc2Threads
                       : kv8                 ? kTc8Threads
                                             : kTcThreads) /
                      32;
        plan->ring_stages = d256                 ? (kv8 ? T256Cfg<true>::k_stages : T256Cfg<false>::k_stages)
                            : tc_rows == kTc2Rows ? kTc2KStages
                            : kv8                 ? TcCfg<true>::k_stages
                                                  : TcCfg<false>::k_stages;
        plan->blocks_per_sm = 1;
        plan->grid_blocks = (int)((long)Hkv * sp.q_tiles * sp.splits * B);
        plan->smem_bytes = d256                 ? (kv8 ? T2568Smem::dynamic : T256Smem::dynamic)
                           : tc_rows == kTc2Rows ? Tc2Smem::dynamic
                           : kv8                 ? Tc8Smem::dynamic
                                                 : TcSmem::dynamic;
        plan->merge_needed = sp.splits > 1 ? 1 : 0;
        plan->q_tiles = sp.q_tiles;
        plan->rows_per_block = tc_rows;
    }
    return PKV_OK;
}

pkv_status paged_prefill_attn_workspace_size(int B, int Hq, int Hkv, int D, int page_size, int max_pages,
                                             int total_q, int max_q_len, int device, int num_splits, int kv_dtype,
                                             size_t *bytes)
{
    if (!bytes) return PKV_ERR_INVALID_ARG;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return PKV_ERR_CUDA;
    pkv_plan plan;
    const pkv_status st =
        pkv_plan_query_prefill(B, Hq, Hkv, D, page_size, max_pages, total_q, max_q_len, sms, num_splits, kv_dtype,
                               &plan);
    if (st != PKV_OK) return st;
    *bytes = plan.workspace_bytes;
    return PKV_OK;
}

pkv_status split_kv_merge(const float *partial_out, const float *partial_lse, int S, int B, int Hq, int D,
                          pkv_bf16 *out, float *lse, cudaStream_t stream)
{
    if (S <= 0 || B < 0 || Hq <= 0) return PKV_ERR_INVALID_ARG;
    if (D != 64 && D != 128 && D != 256) return PKV_ERR_UNSUPPORTED;
    if (B == 0) return PKV_OK;
    if (!partial_out || !partial_lse || !out) return PKV_ERR_INVALID_ARG;
    if (!aligned16(partial_out) || !aligned16(partial_lse) || !aligned16(out) || (lse && !aligned16(lse)))
        return PKV_ERR_MISALIGNED;
    if ((long)S * B * Hq >= (1l << 31)) return PKV_ERR_INVALID_ARG;
    MergeParams mp;
    mp.part_out = partial_out;
    mp.part_lse = partial_lse;
    mp.seq_lens = nullptr;
    mp.out = reinterpret_cast<__nv_bfloat16 *>(out);
    mp.lse = lse;
    mp.S = S;
    mp.B = B;
    mp.Hq = Hq;
    mp.chunk_tokens = 1;
    mp.max_tokens = 0;
    return launch_merge(D, mp, stream);
}

pkv_status paged_kv_append(const pkv_bf16 *k_new, const pkv_bf16 *v_new, const int32_t *block_table,
                           const int32_t *positions, int B, int Hkv, int D, int page_size, int num_pages,
                           int max_pages, pkv_bf16 *k_cache, pkv_bf16 *v_cache, int *status, cudaStream_t stream)
{
    bool skip = false;
    const pkv_status st = append_checks(k_new, v_new, block_table, positions, B, Hkv, D, page_size, num_pages,
                                        max_pages, k_cache, v_cache, status, &skip);
    if (st != PKV_OK || skip) return st;
    AppendParams ap;
    ap.k_new = reinterpret_cast<const uint4 *>(k_new);
    ap.v_new = reinterpret_cast<const uint4 *>(v_new);
    ap.block_table = block_table;
    ap.positions = positions;
    ap.k_cache = reinterpret_cast<uint4 *>(k_cache);
    ap.v_cache = reinterpret_cast<uint4 *>(v_cache);
    ap.status = status;
    ap.B = B;
    ap.Hkv = Hkv;
    ap.D = D;
    ap.P = page_size;
    ap.log2P = log2_exact(page_size);
    ap.num_pages = num_pages;
    ap.max_pages = max_pages;
    const long units = (long)B * Hkv;
    return launch_kernel(kv_append_kernel, dim3((unsigned)((units + kAppendWarps - 1) / kAppendWarps)),
                         dim3(kAppendWarps * 32), 0, stream, ap) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

pkv_status paged_kv_append_fp8(const pkv_bf16 *k_new, const pkv_bf16 *v_new, const int32_t *block_table,
                               const int32_t *positions, int B, int Hkv, int D, int page_size, int num_pages,
                               int max_pages, uint8_t *k_cache, uint8_t *v_cache, float *k_scale, float *v_scale,
                               int *status, cudaStream_t stream)
{
    bool skip = false;
    const pkv_status st = append_checks(k_new, v_new, block_table, positions, B, Hkv, D, page_size, num_pages,
                                        max_pages, k_cache, v_cache, status, &skip);
    if (st != PKV_OK || skip) return st;
    if (!k_scale || !v_scale) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_scale) || !aligned16(v_scale)) return PKV_ERR_MISALIGNED;
    Fp8AppendParams ap;
    ap.k_new = reinterpret_cast<const uint16_t *>(k_new);
    ap.v_new = reinterpret_cast<const uint16_t *>(v_new);
    ap.block_table = block_table;
    ap.positions = positions;
    ap.k_cache = k_cache;
    ap.v_cache = v_cache;
    ap.k_scale = k_scale;
    ap.v_scale = v_scale;
    ap.status = status;
    ap.B = B;
    ap.Hkv = Hkv;
    ap.P = page_size;
    ap.log2P = log2_exact(page_size);
    ap.num_pages = num_pages;
    ap.max_pages = max_pages;
    const long units = (long)B * Hkv;
    const unsigned grid = (unsigned)((units + kAppendWarps - 1) / kAppendWarps);
    cudaError_t e;
    switch (D) {
        case 64: e = launch_kernel(kv_append_fp8_kernel<64>, dim3(grid), dim3(kAppendWarps * 32), 0, stream, ap); break;
        case 128: e = launch_kernel(kv_append_fp8_kernel<128>, dim3(grid), dim3(kAppendWarps * 32), 0, stream, ap); break;
        case 256: e = launch_kernel(kv_append_fp8_kernel<256>, dim3(grid), dim3(kAppendWarps * 32), 0, stream, ap); break;
        default: return PKV_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_check_status(const void *workspace, cudaStream_t stream, int *device_status)
{
    if (!workspace || !device_status) return PKV_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return PKV_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return PKV_ERR_CUDA;
    *device_status = v;
    return PKV_OK;
}

pkv_status pkv_reset_status(void *workspace, cudaStream_t stream)
{
    if (!workspace) return PKV_ERR_INVALID_ARG;
    return cudaMemsetAsync(workspace, 0, sizeof(int), stream) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_selftest_wait_timeout(void *workspace, unsigned timeout_us, cudaStream_t stream)
{
    if (!workspace) return PKV_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return PKV_ERR_MISALIGNED;
    if (timeout_us == 0 || timeout_us > 10000000u) return PKV_ERR_INVALID_ARG;
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(static_cast<int *>(workspace),
                                                        (unsigned long long)timeout_us * 1000ull);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode with library-owned scratch, for callers that cannot allocate device
// memory.
//
// Some callers cannot call cudaMalloc at the point where they run attention:
// code running under an allocator that forbids new device allocations (for
// example a serving loop whose memory pool is sized and frozen at start-up),
// plugins that are handed only the tensors of one step, or hosts that do not
// link the CUDA runtime allocator at all.  For them the split partials and the
// status word live in one fixed file-scope device array instead of a
// caller-provided workspace.  Every GPU that loads this library holds that
// array (kStaticScratchBytes) until the process exits.
//
// The array's name is only a host-side stand-in for the device variable, so
// its device address is looked up with cudaGetSymbolAddress, once per device,
// with that device current, on the first call on that device, and kept for the
// life of the process (not refreshed after cudaDeviceReset, which would leave it
// stale).  Make that first call before any stream capture.  All calls share the
// array and it
// keeps the previous call's contents: each call clears the status word before
// its kernels run, and calls that overlap on the GPU (different streams, or
// different host threads, without ordering) race on it.
// ---------------------------------------------------------------------------

namespace pkv {
namespace {

constexpr size_t kStaticScratchBytes = 32u << 20;  // 32 MiB per device
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_ptr[64] = {};

pkv_status static_scratch_for_current_device(int *device, void **ptr)
{
    if (cudaGetDevice(device) != cudaSuccess) return PKV_ERR_CUDA;
    if (*device < 0 || *device >= 64) return PKV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[*device]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return PKV_ERR_CUDA;
        g_scratch_ptr[*device] = p;
    }
    *ptr = g_scratch_ptr[*device];
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status paged_decode_attn_static_scratch(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                                                       const pkv_bf16 *v_cache, const int32_t *block_table,
                                                       const int32_t *seq_lens, int B, int Hq, int Hkv, int D,
                                                       int page_size, int num_pages, int max_pages, float scale,
                                                       pkv_bf16 *out, float *lse, int *device_status,
                                                       cudaStream_t stream)
{
    // Every host-side check of the workspace entry point first (its workspace is the library's
    // own array), so a rejected call touches neither the GPU nor the scratch.
    bool nothing_to_do = false;
    const pkv_status args_ok =
        pkv::check_decode_args(q, k_cache, v_cache, pkv::Fp8Scales{}, block_table, seq_lens, B, Hq, Hkv, D,
                               page_size, num_pages, max_pages, scale, out, lse, nullptr, true, 0,
                               &nothing_to_do);
    if (args_ok != PKV_OK || nothing_to_do) return args_ok;
    if (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u)) return PKV_ERR_MISALIGNED;

    int device = 0, sms = 0;
    pkv_status st = current_device_sms(&device, &sms);
    if (st != PKV_OK) return st;
    pkv_plan plan;
    st = make_plan(B, Hq, Hkv, D, page_size, max_pages, sms, 0, &plan, false, 0, 0, cluster_merge_enabled());
    if (st != PKV_OK) return st;
    if (plan.workspace_bytes > kStaticScratchBytes) return PKV_ERR_WORKSPACE_TOO_SMALL;

    void *scratch = nullptr;
    st = static_scratch_for_current_device(&device, &scratch);
    if (st != PKV_OK) return st;
    // The status word and the split-completion counters must start at zero (a previous
    // call that gave up part-way could have left a counter raised); the partials are
    // fully written before they are read.
    const size_t zero_bytes =
        workspace_layout(plan.num_splits, (size_t)B * Hkv * plan.q_tiles, (size_t)B * Hq, D).part_lse;
    if (cudaMemsetAsync(scratch, 0, zero_bytes, stream) != cudaSuccess) return PKV_ERR_CUDA;
    st = paged_decode_attn(q, k_cache, v_cache, block_table, seq_lens, B, Hq, Hkv, D, page_size, num_pages,
                           max_pages, scale, out, lse, scratch, kStaticScratchBytes, stream);
    if (st != PKV_OK) return st;
    if (device_status &&
        cudaMemcpyAsync(device_status, scratch, sizeof(int), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}
