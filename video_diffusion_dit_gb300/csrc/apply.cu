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
// Persistent: each CTA owns a contiguous range of 128-token tiles in (head, tile) order.
// Warp 0 streams Q tiles with TMA (two 64-column boxes, 128-byte swizzle = K-major MMA
// layout) and, when the head changes, bulk-copies that head's KV image (three BF16 terms
// KV = hi + mid + lo, already in the swizzled K-major B layout) into shared memory.
// Warp 1 issues, per tile, 3 terms x (Dpad / 16) MMAs of 128 x D x 16 into one of two TMEM
// accumulators.  Warps 2..5 read the accumulator (one token row per thread), multiply by
// the reciprocal denominator and write 32-row boxes through swizzled staging with TMA
// stores.  BF16 x BF16 products are exact in FP32 and the three terms carry 24 bits of
// KV, so the result has FP32-class accuracy (the tier's second GEMM "stays FP32").
constexpr int kApplyStagesPlain = 3;
// The fused path spends shared memory on rotation-table rows instead: fewer Q stages and
// epilogue staging buffers.
#ifndef LA_FUSED_Q_STAGES
#define LA_FUSED_Q_STAGES 2
#endif
#ifndef LA_FUSED_OUT_BUFS
#define LA_FUSED_OUT_BUFS 1
#endif
#ifndef LA_FUSED_TAB_ROWS_MAX
#define LA_FUSED_TAB_ROWS_MAX 64
#endif
constexpr int kApplyStagesFused = LA_FUSED_Q_STAGES;
constexpr int kOutBufsFused = LA_FUSED_OUT_BUFS;
constexpr int kApplyThreads = 192;
constexpr int kApplyThreadsFused = 448;  // + warps 6..13: the producer-step transform
constexpr int kApplyTransformThreads = 256;
constexpr uint32_t kQAtomBytes = kApplyTile * 128;  // 128 token rows x 128 bytes
constexpr uint32_t kOutBoxBytes = 32 * 128;         // 32 rows x 128 bytes

// Fused path: a ring of two slots, each holding the rotation-table rows (cos, then sin) of
// tab_rows consecutive tokens: half a tile where that fits in shared memory, else a quarter.
constexpr uint32_t kSmemLimit = 232448;

// Q stages: a one-atom tile (D <= 64) is half the bytes, so twice the stages keep as many
// bytes in flight.
__host__ __device__ constexpr int apply_stages(int nbox, bool fused) {
    return fused ? (nbox == 1 ? 2 * kApplyStagesFused : kApplyStagesFused)
                 : (nbox == 1 ? 2 * kApplyStagesPlain : kApplyStagesPlain);
}
constexpr uint32_t kApplyBarBytes = 512;  // mbarriers, TMEM address, abort flag

__host__ __device__ constexpr uint32_t apply_smem_bytes_with(int head_dim, bool fused, int tab_rows) {
    const uint32_t nbox = head_dim_atoms(head_dim);
    return static_cast<uint32_t>(kv_image_bytes(head_dim)) + apply_stages(nbox, fused) * nbox * kQAtomBytes +
           4 * (fused ? kOutBufsFused : 2) * kOutBoxBytes +
           (fused ? 2u * tab_rows * (head_dim / 2) * 4u * 2u : 0u) + kApplyBarBytes +
           (fused ? 2 * kApplyTile * 4 : 0) + 1024;
}
__host__ __device__ constexpr int apply_tab_rows(int head_dim) {
    return apply_smem_bytes_with(head_dim, true, LA_FUSED_TAB_ROWS_MAX) <= kSmemLimit ? LA_FUSED_TAB_ROWS_MAX
                                                                                       : LA_FUSED_TAB_ROWS_MAX / 2;
}
__host__ __device__ constexpr uint32_t apply_smem_bytes(int head_dim, bool fused) {
    return apply_smem_bytes_with(head_dim, fused, fused ? apply_tab_rows(head_dim) : 0);
}
// The largest head dim must fit, with whole 16-row groups of table rows per slot.
static_assert(apply_smem_bytes(128, true) <= kSmemLimit && apply_smem_bytes(128, false) <= kSmemLimit &&
                  apply_smem_bytes(64, true) <= kSmemLimit && apply_smem_bytes(64, false) <= kSmemLimit,
              "apply layout exceeds shared memory");
static_assert(apply_tab_rows(128) >= 16 && apply_tab_rows(16) % 16 == 0, "table slots must hold 16-row groups");

template <int NBOX, bool OUT_BF16, bool FUSED>
__global__ void __launch_bounds__(FUSED ? kApplyThreadsFused : kApplyThreads, 1)
    apply_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_out,
                    const uint8_t* __restrict__ kv_image, const float* __restrict__ den, int heads, int n_tokens,
                    int head_dim, int tiles_per_head, int token_major, int* status, const ProducerArgs pa) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);

    constexpr int kApplyStages = apply_stages(NBOX, FUSED);
    constexpr uint32_t kOutBufs = FUSED ? kOutBufsFused : 2u;  // staging buffers per epilogue warp
    const uint32_t img_bytes = 3u * NBOX * head_dim * 128u;
    const uint32_t term_bytes = NBOX * head_dim * 128u;
    const int tab_rows = FUSED ? apply_tab_rows(head_dim) : kApplyTile;  // tokens per table slot
    const uint32_t tab_subs = kApplyTile / tab_rows;                     // table slots per tile
    const uint32_t tab_slot = FUSED ? static_cast<uint32_t>(tab_rows) * (head_dim / 2) * 4u * 2u : 0u;
    const uint32_t b_smem = base;
    const uint32_t q_smem = b_smem + img_bytes;
    const uint32_t o_smem = q_smem + kApplyStages * NBOX * kQAtomBytes;
    const uint32_t tab_smem = o_smem + 4 * kOutBufs * kOutBoxBytes;
    const uint32_t bar_off = tab_smem + 2 * tab_slot - base;
    const uint32_t bars = base + bar_off;
    const uint32_t q_full0 = bars;                        // [kApplyStages]
    const uint32_t q_empty0 = bars + 8u * kApplyStages;   // [kApplyStages]
    const uint32_t acc_full0 = bars + 16u * kApplyStages; // [2]
    const uint32_t acc_empty0 = acc_full0 + 16u;          // [2]
    const uint32_t b_full = acc_empty0 + 16u;
    const uint32_t b_empty = b_full + 8u;
    const uint32_t drain_bar = b_empty + 8u;
    const uint32_t q_ready0 = drain_bar + 8u;             // [kApplyStages] (fused: tile transformed)
    const uint32_t den_full0 = q_ready0 + 8u * kApplyStages;  // [2] (fused: row denominators written)
    const uint32_t den_empty0 = den_full0 + 16u;          // [2] (fused: row denominators read)
    const uint32_t tab_full0 = den_empty0 + 16u;          // [2] (fused: half-tile table rows landed)
    const uint32_t tab_empty0 = tab_full0 + 16u;          // [2] (fused: half-tile table rows used)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + bar_off + kApplyBarBytes - 64);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + bar_off + kApplyBarBytes - 56);
    float* den_s = reinterpret_cast<float*>(base_ptr + bar_off + kApplyBarBytes);  // fused: [2][kApplyTile]
    const uint32_t mma_ready0 = FUSED ? q_ready0 : q_full0;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Head-major activations: contiguous ranges of the layer's (head, tile) sequence.
    // Token-major: gridDim = k heads, CTA b takes part b % k of head b / k, every head cut
    // at the same tiles, so the CTAs running together read and write the same token rows.
    int t_begin, t_end;
    if (!token_major) {
        const int total = heads * tiles_per_head;
        t_begin = static_cast<int>(static_cast<int64_t>(total) * blockIdx.x / gridDim.x);
        t_end = static_cast<int>(static_cast<int64_t>(total) * (blockIdx.x + 1) / gridDim.x);
    } else {
        const int k = gridDim.x / heads, hb = blockIdx.x / k, g = blockIdx.x % k;
        t_begin = hb * tiles_per_head + static_cast<int>(static_cast<int64_t>(tiles_per_head) * g / k);
        t_end = hb * tiles_per_head + static_cast<int>(static_cast<int64_t>(tiles_per_head) * (g + 1) / k);
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kApplyStages; ++s) {
            mbar_init(q_full0 + 8u * s, 1);
            mbar_init(q_empty0 + 8u * s, 1);
            if (FUSED) mbar_init(q_ready0 + 8u * s, kApplyTransformThreads);
        }
        for (int b = 0; b < 2; ++b) {
            if (FUSED) {
                mbar_init(den_full0 + 8u * b, kApplyTransformThreads);
                mbar_init(den_empty0 + 8u * b, 4);
                mbar_init(tab_full0 + 8u * b, 1);
                mbar_init(tab_empty0 + 8u * b, kApplyTransformThreads);
            }
            mbar_init(acc_full0 + 8u * b, 1);
            mbar_init(acc_empty0 + 8u * b, 4);
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
            const uint64_t pol = policy_evict_first();
            uint32_t it = 0;
            int cur_h = -1, run = -1;
            bool ok = true, b_pending = false;
            uint32_t tab_issued = 0;  // half-tile table loads issued
            for (int t = t_begin; t < t_end; ++t, ++it) {
                const int h = t / tiles_per_head;
                const int n0 = (t % tiles_per_head) * kApplyTile;
                const uint32_t st = it % kApplyStages, ph = (it / kApplyStages) & 1u;
                if (!mbar_wait(q_empty0 + 8u * st, ph ^ 1u, abort_flag, status)) {
                    ok = false;
                    break;
                }
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
                    if (run > 0 && !mbar_wait(b_empty, (run - 1) & 1, abort_flag, status)) {
                        ++it;
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(b_full, img_bytes);
                    bulk_load(b_smem, kv_image + static_cast<int64_t>(h) * img_bytes, img_bytes, b_full);
                    b_pending = true;
                }
                if (FUSED) {
                    // The tile's rotation-table rows, tab_rows tokens per slot: rows are
                    // contiguous in the [N][D/2] tables, so a slot is one bulk copy per table,
                    // cut at N.
                    const uint32_t row_bytes = static_cast<uint32_t>(head_dim / 2) * 4u;
                    for (uint32_t hh = 0; hh < tab_subs && ok; ++hh) {
                        const uint32_t i = tab_subs * it + hh;
                        const uint32_t slot = i & 1u, tph = (i >> 1) & 1u;
                        if (!mbar_wait(tab_empty0 + 8u * slot, tph ^ 1u, abort_flag, status)) {
                            ok = false;
                            break;
                        }
                        const int r0 = n0 + static_cast<int>(hh) * tab_rows;
                        const int rows = max(0, min(tab_rows, n_tokens - r0));
                        const uint32_t bytes = static_cast<uint32_t>(rows) * row_bytes;
                        const uint32_t dst = tab_smem + slot * tab_slot;
                        mbar_arrive_expect_tx(tab_full0 + 8u * slot, 2u * bytes);
                        if (rows > 0) {
                            bulk_load(dst, pa.cos + static_cast<int64_t>(r0) * (head_dim / 2), bytes, tab_full0 + 8u * slot);
                            bulk_load(dst + tab_slot / 2, pa.sin + static_cast<int64_t>(r0) * (head_dim / 2), bytes,
                                      tab_full0 + 8u * slot);
                        }
                        tab_issued = i + 1;
                    }
                    if (!ok) {
                        ++it;
                        break;
                    }
                }
            }
            if (!ok) {
                const uint32_t first = it > kApplyStages ? it - kApplyStages : 0;
                for (uint32_t j = first; j < it; ++j)
                    mbar_wait_drain(q_full0 + 8u * (j % kApplyStages), (j / kApplyStages) & 1u);
                if (b_pending) mbar_wait_drain(b_full, run & 1);
                if (FUSED) {
                    const uint32_t tfirst = tab_issued > 2u ? tab_issued - 2u : 0u;  // two slots
                    for (uint32_t j = tfirst; j < tab_issued; ++j) mbar_wait_drain(tab_full0 + 8u * (j & 1u), (j >> 1) & 1u);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            const uint32_t idesc = make_idesc_bf16_f32(128, head_dim, false, false);
            uint32_t it = 0;
            int cur_h = -1, run = -1;
            for (int t = t_begin; t < t_end; ++t, ++it) {
                const int h = t / tiles_per_head;
                const uint32_t lt = static_cast<uint32_t>(t - t_begin);
                if (h != cur_h) {
                    if (run >= 0) mma_commit(b_empty);  // old image free once its MMAs are done
                    ++run;
                    cur_h = h;
                    if (!mbar_wait(b_full, run & 1, abort_flag, status)) break;
                    tc_fence_after();
                }
                const uint32_t buf = lt & 1u;
                if (!mbar_wait(acc_empty0 + 8u * buf, ((lt >> 1) & 1u) ^ 1u, abort_flag, status)) break;
                tc_fence_after();
                const uint32_t st = it % kApplyStages, ph = (it / kApplyStages) & 1u;
                if (!mbar_wait(mma_ready0 + 8u * st, ph, abort_flag, status)) break;
                tc_fence_after();
                const uint32_t d = tmem + buf * 128u;
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
    } else if (FUSED && warp >= 6) {
        // ---------------- producer-step transform of the Q tiles (fused path)
        // Thread (chunk c, row group rg) takes columns 8c..8c+7 of rows rg, rg+16, ..., rg+112:
        // ReLU, dot with the head's column sums of relu(K) (the normaliser), then the rotation
        // (binary32 products and sum in a fixed order, rounded once to BF16).  The 16 threads of
        // a row add their dot products in a fixed butterfly; the row's denominator goes to
        // den_s for the epilogue.  Table rows come from the half-tile slots the producer fills.
        const int u = threadIdx.x - 192;
        const int c = u & 15, rg = u >> 4;
        const bool live = 8 * c < head_dim;
        const uint32_t row_bytes = static_cast<uint32_t>(head_dim / 2) * 4u;
        uint64_t ks[4];  // the head's column sums in rope_chunk's activation order
        int cur_h = -1;
        uint32_t it = 0;
        for (int t = t_begin; t < t_end; ++t, ++it) {
            const int h = t / tiles_per_head;
            const int n0 = (t % tiles_per_head) * kApplyTile;
            const uint32_t lt = static_cast<uint32_t>(t - t_begin);
            if (h != cur_h) {
                if (cur_h < 0) grid_dependency_wait();  // the column sums come from the reduction
                cur_h = h;
                const float* kh = pa.ksum + h * head_dim + 8 * c;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int col = e < 2 ? 4 * e : 4 * (e - 2) + 1;
                    ks[e] = live ? f32x2_pack(kh[col], kh[col + 2]) : 0ull;
                }
            }
            const uint32_t st = it % kApplyStages, ph = (it / kApplyStages) & 1u;
            const uint32_t buf = lt & 1u;
            if (!mbar_wait(q_full0 + 8u * st, ph, abort_flag, status)) break;
            if (!mbar_wait(den_empty0 + 8u * buf, ((lt >> 1) & 1u) ^ 1u, abort_flag, status)) break;
            uint8_t* atom = base_ptr + (q_smem - base) + (st * NBOX + (c >> 3)) * kQAtomBytes;
            bool ok = true;
            const int kper = tab_rows / 16;  // this thread's rows per slot (rows rg + 16 k)
            for (uint32_t hh = 0; hh < tab_subs; ++hh) {
                const uint32_t i = tab_subs * it + hh;
                const uint32_t slot = i & 1u;
                if (!(ok = mbar_wait(tab_full0 + 8u * slot, (i >> 1) & 1u, abort_flag, status))) break;
                const uint8_t* tab = base_ptr + (tab_smem - base) + slot * tab_slot + 16 * c;
                for (int k = kper * static_cast<int>(hh); k < kper * static_cast<int>(hh + 1); ++k) {
                    const int r = rg + 16 * k;
                    const int n = n0 + r;
                    float part = 0.f;
                    if (live && n < n_tokens) {
                        const uint32_t tr = static_cast<uint32_t>(r - static_cast<int>(hh) * tab_rows) * row_bytes;
                        const float4 c4 = *reinterpret_cast<const float4*>(tab + tr);
                        const float4 s4 = *reinterpret_cast<const float4*>(tab + tab_slot / 2 + tr);
                        uint4* cell = reinterpret_cast<uint4*>(atom + r * 128 + (((c & 7) ^ (r & 7)) << 4));
                        uint4 w = *cell;
                        uint64_t a0[2], a1[2];
                        rope_chunk(w, c4, s4, a0, a1);
                        uint64_t d2 = f32x2_mul(a0[0], ks[0]);
                        d2 = f32x2_fma(a0[1], ks[1], d2);
                        d2 = f32x2_fma(a1[0], ks[2], d2);
                        d2 = f32x2_fma(a1[1], ks[3], d2);
                        float d0, d1;
                        f32x2_unpack(d2, d0, d1);
                        part = d0 + d1;
                        *cell = w;
                    }
                    part += __shfl_xor_sync(0xffffffffu, part, 8);
                    part += __shfl_xor_sync(0xffffffffu, part, 4);
                    part += __shfl_xor_sync(0xffffffffu, part, 2);
                    part += __shfl_xor_sync(0xffffffffu, part, 1);
                    if (c == 0) den_s[buf * kApplyTile + r] = part + kDenEps;
                }
                mbar_arrive(tab_empty0 + 8u * slot);
            }
            if (!ok) break;
            fence_proxy_async_smem();
            mbar_arrive(q_ready0 + 8u * st);
            mbar_arrive(den_full0 + 8u * buf);
        }
    } else if (!FUSED || warp < 6) {
        // ---------------- epilogue: warp (q = warp % 4) owns TMEM lanes / tile rows 32q..32q+31
        const int q = warp & 3;
        const uint32_t stage0 = o_smem + static_cast<uint32_t>(warp - 2) * kOutBufs * kOutBoxBytes;
        uint32_t nstore = 0;
        const uint64_t spol = policy_evict_first();
        constexpr int kCols = OUT_BF16 ? 64 : 32;  // columns per 128-byte box row
        const int groups = (head_dim + kCols - 1) / kCols;
        for (int t = t_begin; t < t_end; ++t) {
            const int h = t / tiles_per_head;
            const int n0 = (t % tiles_per_head) * kApplyTile;
            const uint32_t lt = static_cast<uint32_t>(t - t_begin);
            const int row0 = n0 + 32 * q;
            const int row = row0 + lane;
            const uint32_t buf = lt & 1u;
            float dv = 1.0f;
            if (FUSED) {
                if (!mbar_wait(den_full0 + 8u * buf, (lt >> 1) & 1u, abort_flag, status)) break;
                dv = den_s[buf * kApplyTile + 32 * q + lane];
                __syncwarp();
                if (lane == 0) mbar_arrive(den_empty0 + 8u * buf);
            } else if (row < n_tokens) {
                dv = den[static_cast<int64_t>(h) * n_tokens + row];
            }
            const float rcp = __frcp_rn(dv);
            if (!mbar_wait(acc_full0 + 8u * buf, (lt >> 1) & 1u, abort_flag, status)) break;
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * 128u;
            // A warp whose 32 rows all lie past the end of the head (ragged last tile) has
            // nothing to store.  It must not touch its staging buffers either: every buffer
            // write is paired with one committed store, which is what lets wait_group.read 1
            // guarantee the buffer's previous store has finished reading it.
            const int live_groups = row0 < n_tokens ? groups : 0;
            for (int g = 0; g < live_groups; ++g) {
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

template <int NBOX, bool BF16, bool FUSED>
cudaError_t launch_tc(const CUtensorMap& tm_q, const CUtensorMap& tm_out, const uint8_t* img, const float* den,
                      int heads, int n_tokens, int head_dim, bool token_major, int grid, int* status,
                      cudaStream_t stream, const ProducerArgs& pa) {
    const uint32_t smem = apply_smem_bytes(head_dim, FUSED);
    cudaError_t e = cudaFuncSetAttribute(apply_tc_kernel<NBOX, BF16, FUSED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int tph = (n_tokens + kApplyTile - 1) / kApplyTile;
    return launch_overlapped(apply_tc_kernel<NBOX, BF16, FUSED>, dim3(grid),
                             dim3(FUSED ? kApplyThreadsFused : kApplyThreads), smem, stream, tm_q, tm_out, img, den,
                             heads, n_tokens, head_dim, tph, token_major ? 1 : 0, status, pa);
}

template <int NBOX, bool BF16>
cudaError_t launch_tc_any(const CUtensorMap& tm_q, const CUtensorMap& tm_out, const uint8_t* img, const float* den,
                          int heads, int n_tokens, int head_dim, bool token_major, int grid, int* status,
                          cudaStream_t stream, const ProducerArgs* producer) {
    if (producer)
        return launch_tc<NBOX, BF16, true>(tm_q, tm_out, img, den, heads, n_tokens, head_dim, token_major, grid,
                                           status, stream, *producer);
    const ProducerArgs none{nullptr, nullptr, nullptr, nullptr, 0};
    return launch_tc<NBOX, BF16, false>(tm_q, tm_out, img, den, heads, n_tokens, head_dim, token_major, grid, status,
                                        stream, none);
}

}  // namespace

cudaError_t launch_apply_tc(const CUtensorMap& tm_q, const CUtensorMap& tm_out, const uint8_t* kv_image,
                            const float* den, int heads, int64_t n_tokens, int head_dim, bool out_bf16,
                            bool token_major, int grid, int* status, cudaStream_t stream,
                            const ProducerArgs* producer) {
    const int n = static_cast<int>(n_tokens);
    const int tph = (n + kApplyTile - 1) / kApplyTile;
    const int total = heads * tph;
    if (grid > total) grid = total;
    if (token_major) {  // a whole number of CTAs per head (see the kernel's schedule)
        const int k = std::max(1, std::min(grid / heads, tph));
        grid = k * heads;
    }
    const bool one = head_dim_atoms(head_dim) == 1;
    if (one)
        return out_bf16 ? launch_tc_any<1, true>(tm_q, tm_out, kv_image, den, heads, n, head_dim, token_major, grid, status, stream, producer)
                        : launch_tc_any<1, false>(tm_q, tm_out, kv_image, den, heads, n, head_dim, token_major, grid, status, stream, producer);
    return out_bf16 ? launch_tc_any<2, true>(tm_q, tm_out, kv_image, den, heads, n, head_dim, token_major, grid, status, stream, producer)
                    : launch_tc_any<2, false>(tm_q, tm_out, kv_image, den, heads, n, head_dim, token_major, grid, status, stream, producer);
}

}  // namespace la
