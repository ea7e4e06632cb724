// Second GEMM + normalisation of SANA-Video linear attention:
//     out[h][n][:] = (Q_rot[h][n][:] . KV[h]) / den[h][n]
//
// Page "PR #35728 完整报告 - [diffusion] Accelerate SANA-Video linear attention in
// quality=high", 关键源码片段: (scores @ query_rotate.float()) * normalizer, and the
// page's note that the second GEMM stays FP32 in both tiers.  The page multiplies by a
// precomputed reciprocal; here each token's denominator is turned into a correctly rounded
// reciprocal once and the row is multiplied by it (within 1 ulp of a true division).
#include <cuda_bf16.h>

#include <algorithm>

#include "lin_attn_internal.cuh"
#include "ptx.cuh"

namespace la {
namespace {

// ============================================================================ tensor cores
// Persistent: each CTA owns a contiguous range of 128-token tiles in (head, tile) order
// (token-major activations: a chunk of the body + tail split).  Warp 0 streams Q tiles with
// TMA (two 64-column boxes, 128-byte swizzle = K-major MMA layout) and, when the head
// changes, bulk-copies that head's KV image (three BF16 terms KV = hi + mid + lo, already in
// the swizzled K-major B layout) into shared memory.  Warp 1 issues, per tile, 3 terms x
// (Dpad / 16) MMAs of 128 x D x 16 into one of the TMEM accumulators (two, or four when
// D <= 64).  Warps 2..9 read the accumulator (one token row per thread; two warps per TMEM
// lane quarter, each with half of the tile's column groups, or alternate tiles where there
// is one group), multiply by the reciprocal denominator (loaded a tile ahead) and write
// 32-row boxes through swizzled staging with TMA stores (stage and staging-buffer counts in
// apply_stages / apply_out_bufs).  BF16 x BF16 products are exact in FP32 and the three
// terms carry 24 bits of KV, so the result has FP32-class accuracy (the tier's second GEMM
// "stays FP32").
constexpr int kApplyEpiWarps = 8;
constexpr int kApplyThreads = 32 * (2 + kApplyEpiWarps);
constexpr uint32_t kQAtomBytes = kApplyTile * 128;  // 128 token rows x 128 bytes
constexpr uint32_t kOutBoxBytes = 32 * 128;         // 32 rows x 128 bytes
constexpr uint32_t kApplyBarBytes = 512;            // mbarriers, TMEM address, abort flag
constexpr uint32_t kSmemLimit = 232448;

// Shared memory beside the KV image goes to Q stages and output staging.  A one-atom tile
// (D <= 64) is half the bytes, so it gets twice the stages.  With FP32 output and two atoms
// the output is twice the bytes of Q and the staging is what paces the epilogue: two Q
// stages and two staging buffers per warp (0.4055 -> 0.3874 ms at 720p) rather than three
// and one; BF16 output keeps three and one (two and two: 0.2780 -> 0.2805 ms).  At D <= 64
// a third staging buffer per warp changed nothing (0.4118 / 0.4121 ms).
__host__ __device__ constexpr int apply_stages(int nbox, bool bf16) { return nbox == 1 ? 6 : (bf16 ? 3 : 2); }
__host__ __device__ constexpr uint32_t apply_out_bufs(int nbox, bool bf16) {
    return nbox == 1 ? 2u : (bf16 ? 1u : 2u);
}

__host__ __device__ constexpr uint32_t apply_smem_bytes(int head_dim, bool bf16) {
    return static_cast<uint32_t>(kv_image_bytes(head_dim)) +
           apply_stages(head_dim_atoms(head_dim), bf16) * head_dim_atoms(head_dim) * kQAtomBytes +
           kApplyEpiWarps * apply_out_bufs(head_dim_atoms(head_dim), bf16) * kOutBoxBytes + kApplyBarBytes + 1024;
}
static_assert(apply_smem_bytes(128, false) <= kSmemLimit && apply_smem_bytes(64, false) <= kSmemLimit &&
                  apply_smem_bytes(128, true) <= kSmemLimit && apply_smem_bytes(64, true) <= kSmemLimit,
              "apply layout exceeds shared memory");

template <int NBOX, bool OUT_BF16>
__global__ void __launch_bounds__(kApplyThreads, 1)
    apply_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_out,
                    const uint8_t* kv_image, const float* __restrict__ den, int heads, int n_tokens,
                    int head_dim, const TileSplit sp, int token_major, int* status, uint64_t wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);

    constexpr int kApplyStages = apply_stages(NBOX, OUT_BF16);
    const uint32_t img_bytes = 3u * NBOX * head_dim * 128u;
    const uint32_t term_bytes = NBOX * head_dim * 128u;
    const uint32_t b_smem = base;
    const uint32_t q_smem = b_smem + img_bytes;
    const uint32_t o_smem = q_smem + kApplyStages * NBOX * kQAtomBytes;
    constexpr uint32_t kOutBufs = apply_out_bufs(NBOX, OUT_BF16);
    const uint32_t bar_off = o_smem + kApplyEpiWarps * kOutBufs * kOutBoxBytes - base;
    const uint32_t bars = base + bar_off;
    const uint32_t q_full0 = bars;                        // [kApplyStages]
    const uint32_t q_empty0 = bars + 8u * kApplyStages;   // [kApplyStages]
    // TMEM accumulators (N = D columns each, in 256 allocated columns): two of 128 columns, or
    // four of 64 when D <= 64, so that the MMA can run further ahead of the epilogue there.
    constexpr uint32_t kAcc = NBOX == 1 ? 4u : 2u;
    constexpr uint32_t kAccCols = 256u / kAcc;
    static_assert((2 * kApplyStages + 2 * kAcc + 3) * 8 <= kApplyBarBytes - 64, "barriers overlap the TMEM address slot");
    const uint32_t acc_full0 = bars + 16u * kApplyStages; // [kAcc]
    const uint32_t acc_empty0 = acc_full0 + 8u * kAcc;    // [kAcc]
    const uint32_t b_full = acc_empty0 + 8u * kAcc;
    const uint32_t b_empty = b_full + 8u;
    const uint32_t drain_bar = b_empty + 8u;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + bar_off + kApplyBarBytes - 64);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + bar_off + kApplyBarBytes - 56);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Head-major activations: contiguous ranges of the layer's (head, tile) sequence (sp has
    // no tail: tile t is tile t % T of head t / T).  Token-major: the CTAs are the chunks of
    // the body + tail split sp (every head's body cut at the same tiles, so the CTAs running
    // together read and write the same token rows; the spare CTAs share the tails).
    int t_begin, t_end;
    if (!token_major) {
        const int total = heads * static_cast<int>(sp.tiles_per_head);
        t_begin = static_cast<int>(static_cast<int64_t>(total) * blockIdx.x / gridDim.x);
        t_end = static_cast<int>(static_cast<int64_t>(total) * (blockIdx.x + 1) / gridDim.x);
    } else {
        t_begin = static_cast<int>(split_begin(sp, blockIdx.x));
        t_end = static_cast<int>(split_begin(sp, blockIdx.x + 1));
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kApplyStages; ++s) {
            mbar_init(q_full0 + 8u * s, 1);
            mbar_init(q_empty0 + 8u * s, 1);
        }
        for (uint32_t b = 0; b < kAcc; ++b) {
            mbar_init(acc_full0 + 8u * b, 1);
            mbar_init(acc_empty0 + 8u * b, kApplyEpiWarps);
        }
        mbar_init(b_full, 1);
        mbar_init(b_empty, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), 256);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_out);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // The next layer call's first kernel waits for this grid to complete before it touches
    // anything, so it may be scheduled right away.
    grid_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- producer
            // Q tiles are inputs of the call and may be fetched before the reduction that
            // produces the KV image has finished; the image is loaded only after the wait.
            bool waited = false;
            // Token-major Q rows share DRAM granules with the neighbouring heads' rows, which
            // other CTAs read at about the same time: those lines stay at normal priority.
            const uint64_t pol = token_major ? policy_evict_normal() : policy_evict_first();
            uint32_t it = 0;
            int cur_h = -1, run = -1;
            bool b_pending = false;
            for (int t = t_begin; t < t_end; ++t, ++it) {
                int h, tile;
                split_tile32(sp, t, h, tile);
                const int n0 = tile * kApplyTile;
                const uint32_t st = it % kApplyStages, ph = (it / kApplyStages) & 1u;
                if (!mbar_wait(q_empty0 + 8u * st, ph ^ 1u, abort_flag, status, wait_ns)) break;
                mbar_arrive_expect_tx(q_full0 + 8u * st, NBOX * kQAtomBytes);
#pragma unroll
                for (int x = 0; x < NBOX; ++x)
                    tma_load_3d_hint(q_smem + (st * NBOX + x) * kQAtomBytes, &tm_q, q_full0 + 8u * st, 64 * x,
                                     token_major ? h : n0, token_major ? n0 : h, pol);
                if (h != cur_h) {
                    if (!waited) {
                        grid_dependency_wait();
                        waited = true;
                    }
                    ++run;
                    cur_h = h;
                    if (run > 0 && !mbar_wait(b_empty, (run - 1) & 1, abort_flag, status, wait_ns)) {
                        ++it;  // this tile's Q load was issued
                        --run;  // ... but not this head's image
                        break;
                    }
                    mbar_arrive_expect_tx(b_full, img_bytes);
                    bulk_load(b_smem, kv_image + static_cast<int64_t>(h) * img_bytes, img_bytes, b_full);
                    b_pending = true;
                }
            }
            // Let the copies already issued land before shared memory goes away: the MMA
            // issuer waits for all of them unless some role gave up, in which case nothing
            // else would.  (`it` Q loads were issued, only the last kApplyStages can be
            // pending; image `run` is the only image load that can be.)
            const uint32_t first = it > kApplyStages ? it - kApplyStages : 0;
            for (uint32_t j = first; j < it; ++j)
                mbar_wait_drain(q_full0 + 8u * (j % kApplyStages), (j / kApplyStages) & 1u);
            if (b_pending) mbar_wait_drain(b_full, run & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            const uint32_t idesc = make_idesc_bf16_f32(128, head_dim, false, false);
            uint32_t it = 0;
            int cur_h = -1, run = -1;
            for (int t = t_begin; t < t_end; ++t, ++it) {
                int h, tile;
                split_tile32(sp, t, h, tile);
                const uint32_t lt = static_cast<uint32_t>(t - t_begin);
                if (h != cur_h) {
                    if (run >= 0) mma_commit(b_empty);  // old image free once its MMAs are done
                    ++run;
                    cur_h = h;
                    if (!mbar_wait(b_full, run & 1, abort_flag, status, wait_ns)) break;
                    tc_fence_after();
                }
                const uint32_t buf = lt % kAcc;
                if (!mbar_wait(acc_empty0 + 8u * buf, ((lt / kAcc) & 1u) ^ 1u, abort_flag, status, wait_ns)) break;
                tc_fence_after();
                const uint32_t st = it % kApplyStages, ph = (it / kApplyStages) & 1u;
                if (!mbar_wait(q_full0 + 8u * st, ph, abort_flag, status, wait_ns)) break;
                tc_fence_after();
                const uint32_t d = tmem + buf * kAccCols;
                const uint32_t qa = q_smem + st * NBOX * kQAtomBytes;
                // Smallest term first; every product is exact, the accumulator is FP32.
#pragma unroll
                for (int term = 2; term >= 0; --term) {
#pragma unroll
                    for (int ks = 0; ks < 4 * NBOX; ++ks) {
                        const uint32_t x = ks >> 2, off = (ks & 3) * 32u;
                        const uint64_t ad = make_smem_desc(qa + x * kQAtomBytes + off, 16u, 1024u, kSwizzle128B);
                        const uint64_t bd = make_smem_desc(b_smem + term * term_bytes + x * head_dim * 128u + off,
                                                           16u, 1024u, kSwizzle128B);
                        mma_bf16(d, ad, bd, idesc, (term != 2 || ks != 0) ? 1u : 0u);
                    }
                }
                mma_commit(q_empty0 + 8u * st);
                mma_commit(acc_full0 + 8u * buf);
            }
            mma_commit(drain_bar);
            mbar_wait_drain(drain_bar, 0);
        }
    } else {
        // ---------------- epilogue: warp (q = warp % 4) owns TMEM lanes / tile rows 32q..32q+31,
        // half eh = (warp - 2) / 4 of the column groups
        const int q = warp & 3;
        const int eh = (warp - 2) >> 2;
        const uint32_t stage0 = o_smem + static_cast<uint32_t>(warp - 2) * kOutBufs * kOutBoxBytes;
        uint32_t nstore = 0;
        // Token-major output rows share L2 lines with the neighbouring heads' rows (written by
        // other CTAs): normal priority, as for the loads.
        const uint64_t spol = token_major ? policy_evict_normal() : policy_evict_first();
        constexpr int kCols = OUT_BF16 ? 64 : 32;  // columns per 128-byte box row
        const int groups = (head_dim + kCols - 1) / kCols;
        // The two warps of a lane quarter take half of the column groups each; with a single
        // group (BF16 output at D <= 64, FP32 at D <= 32) they take alternate tiles instead.
        const bool by_tile = groups == 1;
        const int g_per = (groups + 1) / 2;
        const int g_lo = by_tile ? 0 : eh * g_per, g_hi = by_tile ? 1 : min(groups, g_lo + g_per);
        auto mine = [&](uint32_t ltile) { return !by_tile || static_cast<int>(ltile & 1u) == eh; };
        // The denominators of this warp's next tile are loaded while the current one is written
        // out, so the load's latency is not on the path from an accumulator landing to its
        // stores (720p apply: FP32 out 0.3877 -> 0.3865 ms, BF16 0.2791 -> 0.2643; D = 64 FP32
        // 0.4110 -> 0.3716).
        auto den_of = [&](int tt) {
            int hh, ti;
            split_tile32(sp, tt, hh, ti);
            const int r = ti * kApplyTile + 32 * q + lane;
            return r < n_tokens ? den[static_cast<int64_t>(hh) * n_tokens + r] : 1.0f;
        };
        float dv_next = t_begin < t_end && mine(0) ? den_of(t_begin) : 1.0f;
        for (int t = t_begin; t < t_end; ++t) {
            int h, tile;
            split_tile32(sp, t, h, tile);
            const int n0 = tile * kApplyTile;
            const uint32_t lt = static_cast<uint32_t>(t - t_begin);
            const int row0 = n0 + 32 * q;
            const uint32_t buf = lt % kAcc;
            const float dv = dv_next;
            if (t + 1 < t_end && mine(lt + 1)) dv_next = den_of(t + 1);
            const float rcp = __frcp_rn(dv);
            if (!mbar_wait(acc_full0 + 8u * buf, (lt / kAcc) & 1u, abort_flag, status, wait_ns)) break;
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * kAccCols;
            // A warp whose 32 rows all lie past the end of the head (ragged last tile) has
            // nothing to store.  It must not touch its staging buffers either: every buffer
            // write is paired with one committed store, which is what lets wait_group.read 1
            // guarantee the buffer's previous store has finished reading it.
            const int live_hi = row0 < n_tokens && mine(lt) ? g_hi : g_lo;
            for (int g = g_lo; g < live_hi; ++g) {
                uint32_t packed[32];
                if (!OUT_BF16) {
                    uint32_t r[32];
                    tmem_ld32_sync(taddr + 32u * g, r);
#pragma unroll
                    for (int e = 0; e < 32; ++e) packed[e] = __float_as_uint(__uint_as_float(r[e]) * rcp);
                } else {
                    uint32_t r[32];
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        tmem_ld32_sync(taddr + 64u * g + 32u * half, r);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const __nv_bfloat162 p = __floats2bfloat162_rn(__uint_as_float(r[2 * e]) * rcp,
                                                                           __uint_as_float(r[2 * e + 1]) * rcp);
                            packed[16 * half + e] = *reinterpret_cast<const uint32_t*>(&p);
                        }
                    }
                }
                const uint32_t sbuf = stage0 + (nstore % kOutBufs) * kOutBoxBytes;
                if (lane == 0) bulk_wait_read<kOutBufs - 1>();
                __syncwarp();
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t addr = sbuf + lane * 128u + ((static_cast<uint32_t>(c) ^ (lane & 7u)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(packed[4 * c]),
                                 "r"(packed[4 * c + 1]), "r"(packed[4 * c + 2]), "r"(packed[4 * c + 3])
                                 : "memory");
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d_hint(&tm_out, sbuf, kCols * g, token_major ? h : row0, token_major ? row0 : h, spol);
                    bulk_commit();
                }
                ++nstore;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty0 + 8u * buf);
        }
        if (lane == 0) bulk_wait<0>();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

template <int NBOX, bool BF16>
cudaError_t launch_tc(const CUtensorMap& tm_q, const CUtensorMap& tm_out, const uint8_t* img, const float* den,
                      int heads, int n_tokens, int head_dim, bool token_major, const TileSplit& sp, int grid,
                      int* status, uint64_t wait_ns, cudaStream_t stream, bool overlap) {
    const uint32_t smem = apply_smem_bytes(head_dim, BF16);
    cudaError_t e = cudaFuncSetAttribute(apply_tc_kernel<NBOX, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_kernel(overlap, apply_tc_kernel<NBOX, BF16>, dim3(grid), dim3(kApplyThreads), smem, stream, tm_q,
                         tm_out, img, den, heads, n_tokens, head_dim, sp, token_major ? 1 : 0, status, wait_ns);
}

}  // namespace

cudaError_t launch_apply_tc(const CUtensorMap& tm_q, const CUtensorMap& tm_out, const uint8_t* kv_image,
                            const float* den, int heads, int64_t n_tokens, int head_dim, bool out_bf16,
                            bool token_major, int grid, int* status, uint64_t wait_ns, cudaStream_t stream,
                            bool overlap) {
    const int n = static_cast<int>(n_tokens);
    const int tph = (n + kApplyTile - 1) / kApplyTile;
    const int total = heads * tph;
    TileSplit sp;
    if (token_major) {  // the CTAs are the chunks of the split (see the kernel's schedule)
        sp = tile_split(heads, tph, grid, kNoPerHeadCap, kApplyMinPart, kApplySwitchCost);
        grid = sp.chunks;
    } else {  // whole heads, no tail: only the tile -> (head, tile) map is used
        sp = tile_split(heads, tph, heads, 1, 0, 0);
        if (grid > total) grid = total;
    }
    const bool one = head_dim_atoms(head_dim) == 1;
#define LA_APPLY(NB, BF) \
    launch_tc<NB, BF>(tm_q, tm_out, kv_image, den, heads, n, head_dim, token_major, sp, grid, status, wait_ns, stream, \
                      overlap)
    if (one) return out_bf16 ? LA_APPLY(1, true) : LA_APPLY(1, false);
    return out_bf16 ? LA_APPLY(2, true) : LA_APPLY(2, false);
#undef LA_APPLY
}

}  // namespace la
