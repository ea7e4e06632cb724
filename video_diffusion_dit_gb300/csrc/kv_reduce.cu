// First GEMM of SANA-Video linear attention: KV[h] = K_rot[h]^T . V[h], reduced over tokens.
//
// Page "PR #35728 完整报告 - [diffusion] Accelerate SANA-Video linear attention in
// quality=high", 关键源码片段: the site runs the first GEMM as a BF16 bmm with FP32
// accumulation/output ('high'); the model's fallback chain upcasts both operands to FP32
// first ('lossless').
//
// Both tiers run on tensor cores: BF16 x BF16 products are exact in FP32, so the first
// GEMM on BF16 operands is the FP32 GEMM on the upcast operands up to rounding; 'lossless'
// promotes the tensor-core sums into FP32 registers four times as often.
//
// Work split (KvPlan, lin_attn_internal.cuh): k chunks per head on the first B of each
// head's 64-token tiles, cut at the same token boundaries for every head, and on long
// sequences the spare chunks (152 - k H) on the remaining tiles of all heads; one CTA per
// chunk.  Each run of a chunk within one head (a "segment") leaves one D x D partial sum;
// kv_finalize adds each head's partials in a fixed pairwise order.  The split depends on
// the shape alone, and so do the order and the result.
#include <cuda_bf16.h>

#include "lin_attn_internal.cuh"
#include "ptx.cuh"

namespace la {
namespace {

// ============================================================================ tensor cores
// Warp roles: warp 0 issues TMA loads, warp 1 issues tcgen05.mma, warps 2..5 drain the
// TMEM accumulator; the fused-producer instantiation adds warps 6..13, which turn each
// loaded K tile into relu(K) rotated (in place) and sum the columns of relu(K).  Per
// stage, one 64-token tile of K and of V is loaded with 128-byte swizzle as
// [token][64 head-dim columns] boxes - exactly the MN-major canonical layout of
// the MMA operands A = K^T (M = head-dim row i) and B = V (N = head-dim column j), with
// K = tokens.  M is always 128 (head dims up to 128; rows i >= D are zero).
constexpr int kKvStages = 6;
constexpr int kKvThreads = 192;
constexpr int kKvTransformThreads = 256;  // warps 6..13: the producer-step transform
constexpr int kKvThreadsFused = 192 + kKvTransformThreads;
static_assert(kKvTransformThreads == 16 * ksum_groups(128) && kKvTransformThreads == 8 * ksum_groups(64) &&
                  kKvTile % ksum_groups(64) == 0 && kKvTile % ksum_groups(128) == 0,
              "transform thread (chunk, row group) covers rows rg + groups k of every tile");
// Tiles per tensor-core sub-chunk before its sum is promoted into FP32 registers: 4 (256
// tokens) in the 'high' tier, 1 (64 tokens) in the 'lossless' tier.
constexpr int kPromoteHigh = 4;
constexpr int kPromoteLossless = 1;
constexpr uint32_t kKvAtomBytes = kKvTile * 128;  // one box: 64 token rows x 128 bytes

template <int NBOX, bool FUSED>
struct KvLayout {
    // The fused path also stages the tile's rows of the two rotation tables (FP32,
    // [64 tokens][D/2], at most 16 KB each) in a ring of their own: the tables mostly come
    // from L2 (every head reads the same rows), K and V from DRAM.  When D > 64 the K/V ring
    // keeps four tiles in flight and the table ring three (a table copy is issued two tiles
    // before its transform); when D <= 64 six and four, since a tile then takes about half
    // the time and the table ring must still cover a copy's ~1.8 us from L2.
    static constexpr int stages = FUSED ? (NBOX == 1 ? 6 : 4) : kKvStages;
    static constexpr int tab_ring = NBOX == 1 ? 4 : 3;  // table slots of the fused kernel
    static constexpr int tab_slots = FUSED ? tab_ring : 0;  // ... and the shared memory they take
    static constexpr uint32_t a_bytes = 2 * kKvAtomBytes;  // A = K^T: 2 atoms cover M = 128
    static constexpr uint32_t b_bytes = NBOX * kKvAtomBytes;
    static constexpr uint32_t tab_bytes = kKvTile * 32 * NBOX * 4;  // one table's rows, D/2 <= 32 NBOX columns
    static constexpr uint32_t stage_bytes = a_bytes + b_bytes;
    static constexpr uint32_t tab_offset = stages * stage_bytes;  // [tab_slots][cos, sin]
    static constexpr uint32_t bar_offset = tab_offset + tab_slots * 2 * tab_bytes;
    static constexpr uint32_t bar_bytes = 512;
    static constexpr uint32_t smem_bytes = bar_offset + bar_bytes + 1024;  // + barriers + alignment slack
    // TMEM: two 128-column accumulators; the fused kernel keeps the segment's running sum in
    // a third region (columns 256..383) instead of registers, which leaves the registers to
    // its transform warps.
    static constexpr uint32_t tmem_cols = FUSED ? 512 : 256;
    static constexpr uint32_t sum_col = 256;
    static_assert(!FUSED || sum_col + 128 <= tmem_cols, "the running sums must fit beside the accumulators");
};

static_assert(KvLayout<2, true>::smem_bytes <= 232448 && KvLayout<2, false>::smem_bytes <= 232448 &&
                  KvLayout<1, true>::smem_bytes <= 232448 && KvLayout<1, false>::smem_bytes <= 232448,
              "KV layout exceeds the 227 KB of shared memory a CTA may use");

// Virtual tiles [t_s, t_e) of the CTA's chunk (see TileSplit), clipped to the launch's heads.
struct ChunkTiles {
    int64_t c, t_s, t_e;
};
__device__ __forceinline__ ChunkTiles chunk_tiles(const KvPlan& plan, const KvLaunch& work) {
    ChunkTiles r;
    const int b = static_cast<int>(blockIdx.x);
    if (b < work.n_body) {
        r.c = work.c_body + b;
        r.t_s = split_begin(plan, r.c);
        r.t_e = split_begin(plan, r.c + 1);
    } else {
        r.c = work.c_tail + (b - work.n_body);
        r.t_s = max(split_begin(plan, r.c), work.tail_lo);
        r.t_e = min(split_begin(plan, r.c + 1), work.tail_hi);
    }
    return r;
}

template <int NBOX, bool FUSED, int PROMOTE>
__global__ void __launch_bounds__(FUSED ? kKvThreadsFused : kKvThreads, 1)
    kv_partial_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         float* __restrict__ partial, int head_dim, const KvPlan plan, const KvLaunch work,
                         int token_major, int* status, uint64_t wait_ns, const ProducerArgs pa,
                         const __grid_constant__ CUtensorMap tm_cos, const __grid_constant__ CUtensorMap tm_sin) {
    using L = KvLayout<NBOX, FUSED>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);

    const uint32_t bars = base + L::bar_offset;
    const uint32_t full0 = bars;                          // [L::stages]
    const uint32_t empty0 = bars + 8u * L::stages;        // [L::stages]
    const uint32_t acc_full0 = bars + 16u * L::stages;    // [2]
    const uint32_t acc_empty0 = acc_full0 + 16u;          // [2]
    const uint32_t drain_bar = acc_empty0 + 16u;
    const uint32_t ready0 = drain_bar + 8u;               // [L::stages] (fused: tile transformed)
    const uint32_t tab_full0 = ready0 + 8u * L::stages;   // [L::tab_slots] (fused: table rows landed)
    const uint32_t tab_empty0 = tab_full0 + 8u * L::tab_slots;  // [L::tab_slots] (... and used)
    static_assert(3 * L::stages * 8 + 40 + 16 * L::tab_slots <= L::bar_bytes - 16,
                  "barriers overlap the TMEM address slot");
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + L::bar_offset + L::bar_bytes - 16);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + L::bar_offset + L::bar_bytes - 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const ChunkTiles ct = chunk_tiles(plan, work);
    // The MMA consumes a stage once it is loaded (full) or, on the fused path, transformed.
    const uint32_t mma_ready0 = FUSED ? ready0 : full0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < L::stages; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, 1);
            if (FUSED) mbar_init(ready0 + 8u * s, kKvTransformThreads);
        }
        for (int s = 0; s < L::tab_slots; ++s) {
            mbar_init(tab_full0 + 8u * s, 1);
            mbar_init(tab_empty0 + 8u * s, kKvTransformThreads);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full0 + 8u * b, 1);
            mbar_init(acc_empty0 + 8u * b, 4);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (NBOX == 1) {
        // Head dim <= 64: the second A atom (rows i = 64..127) is never loaded; zero it once.
        for (uint32_t idx = threadIdx.x; idx < L::stages * (kKvAtomBytes / 16); idx += blockDim.x) {
            const uint32_t st = idx / (kKvAtomBytes / 16), off = idx % (kKvAtomBytes / 16);
            *reinterpret_cast<uint4*>(base_ptr + st * L::stage_bytes + kKvAtomBytes + off * 16) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), L::tmem_cols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        if (FUSED) {
            prefetch_tmap(&tm_cos);
            prefetch_tmap(&tm_sin);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // The prologue above overlaps the previous kernel's tail; K/V, and the partial buffer
    // the previous layer call's reduction reads, are touched only after this.
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- producer: every tile of the chunk, in order
            // Token-major K/V rows share DRAM granules with the neighbouring heads' rows, which
            // other CTAs read at about the same time: those lines stay at normal priority.
            const uint64_t pol = token_major ? policy_evict_normal() : policy_evict_first();
            const uint64_t tab_pol = policy_evict_last();
            uint32_t it = 0, n_tab = 0;  // K/V loads issued; table loads issued (fused)
            // (head, tile) of t, advanced by one per tile and recomputed where a run ends.
            HeadTile ht{0, 0};
            int64_t run_end = ct.t_s;
            for (int64_t t = ct.t_s; t < ct.t_e; ++t, ++it, ++ht.tile) {
                if (t == run_end) {
                    ht = split_tile(plan, t);
                    run_end = split_run_end(plan, t);
                }
                const int h = ht.h;
                const int y = static_cast<int>(ht.tile * kKvTile);
                const int c1 = token_major ? h - work.h0 : y, c2 = token_major ? y : h - work.h0;
                const uint32_t st = it % L::stages, ph = (it / L::stages) & 1u;
                if (!mbar_wait(empty0 + 8u * st, ph ^ 1u, abort_flag, status, wait_ns)) break;
                const uint32_t a = base + st * L::stage_bytes;
                const uint32_t b = a + L::a_bytes;
                mbar_arrive_expect_tx(full0 + 8u * st, 2u * NBOX * kKvAtomBytes);
#pragma unroll
                for (int x = 0; x < NBOX; ++x) {
                    tma_load_3d_hint(a + x * kKvAtomBytes, &tm_k, full0 + 8u * st, 64 * x, c1, c2, pol);
                    tma_load_3d_hint(b + x * kKvAtomBytes, &tm_v, full0 + 8u * st, 64 * x, c1, c2, pol);
                }
                if constexpr (FUSED) {
                    // Rotation-table rows of the tile's tokens (kept in L2: every head re-reads
                    // them), into the table slot the transform of tile it - tab_slots freed.
                    const uint32_t ts = it % L::tab_slots, tpar = (it / L::tab_slots) & 1u;
                    if (!mbar_wait(tab_empty0 + 8u * ts, tpar ^ 1u, abort_flag, status, wait_ns)) {
                        ++it;  // this tile's K/V loads were issued
                        break;
                    }
                    const uint32_t tab = base + L::tab_offset + ts * 2u * L::tab_bytes;
                    mbar_arrive_expect_tx(tab_full0 + 8u * ts, 2u * kKvTile * (head_dim / 2) * 4u);
                    tma_load_2d_hint(tab, &tm_cos, tab_full0 + 8u * ts, 0, y, tab_pol);
                    tma_load_2d_hint(tab + L::tab_bytes, &tm_sin, tab_full0 + 8u * ts, 0, y, tab_pol);
                    ++n_tab;
                }
            }
            // Let the loads already issued land before shared memory goes away: the MMA
            // issuer and the transform wait for all of them unless some role gave up, in which
            // case nothing else would.  (`it` K/V loads and `n_tab` table loads were issued;
            // only the last `stages` / `tab_slots` of each can be pending.)
            const uint32_t first = it > L::stages ? it - L::stages : 0;
            for (uint32_t j = first; j < it; ++j)
                mbar_wait_drain(full0 + 8u * (j % L::stages), (j / L::stages) & 1u);
            if constexpr (FUSED) {
                const uint32_t first_tab = n_tab > L::tab_slots ? n_tab - L::tab_slots : 0;
                for (uint32_t j = first_tab; j < n_tab; ++j)
                    mbar_wait_drain(tab_full0 + 8u * (j % L::tab_slots), (j / L::tab_slots) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            // Each segment (the chunk's tiles of one head) is accumulated in sub-chunks of
            // PROMOTE tiles, alternating between two TMEM accumulators; the epilogue
            // adds every finished sub-chunk into FP32 registers (round-to-nearest), so
            // tensor-core accumulation never runs over more than PROMOTE * 64 tokens.
            constexpr uint32_t idesc = make_idesc_bf16_f32(128, 64 * NBOX, true, true);
            uint32_t it = 0, sub = 0;
            bool ok = true;
            for (int64_t t = ct.t_s; ok && t < ct.t_e;) {
                const int64_t seg_end = min(ct.t_e, split_run_end(plan, t));
                for (int64_t k0 = t; ok && k0 < seg_end; k0 += PROMOTE, ++sub) {
                    const int64_t k1 = min(k0 + PROMOTE, seg_end);
                    const uint32_t buf = sub & 1u;
                    if (!mbar_wait(acc_empty0 + 8u * buf, ((sub >> 1) & 1u) ^ 1u, abort_flag, status, wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + buf * 128u;
                    for (int64_t k = k0; k < k1; ++k, ++it) {
                        const uint32_t st = it % L::stages, ph = (it / L::stages) & 1u;
                        if (!mbar_wait(mma_ready0 + 8u * st, ph, abort_flag, status, wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a = base + st * L::stage_bytes;
                        const uint32_t b = a + L::a_bytes;
#pragma unroll
                        for (int kk = 0; kk < kKvTile / 16; ++kk) {
                            // 16 tokens = 2 groups of 8 rows of 128 B: advance by 2048 B per step.
                            const uint64_t ad = make_smem_desc(a + kk * 2048u, kKvAtomBytes, 1024u, kSwizzle128B);
                            const uint64_t bd = make_smem_desc(b + kk * 2048u, kKvAtomBytes, 1024u, kSwizzle128B);
                            mma_bf16(d, ad, bd, idesc, (k != k0 || kk != 0) ? 1u : 0u);
                        }
                        mma_commit(empty0 + 8u * st);
                    }
                    if (ok) mma_commit(acc_full0 + 8u * buf);
                }
                t = seg_end;
            }
            mma_commit(drain_bar);
            mbar_wait_drain(drain_bar, 0);
        }
    } else if (FUSED && warp >= 6) {
        // ---------------- producer-step transform of the K tiles (fused path)
        constexpr int kCpr = 8 * NBOX;                       // chunk lanes per row
        constexpr int kGroups = kKvTransformThreads / kCpr;  // = ksum_groups(head_dim)
        const int u = threadIdx.x - 192;
        const int c = u % kCpr, rg = u / kCpr;
        const bool live = 8 * c < head_dim;
        const int64_t pairs = head_dim / 2;
        uint32_t it = 0;
        bool ok = true;
        for (int64_t t = ct.t_s; ok && t < ct.t_e;) {
            const int h = split_tile(plan, t).h;
            const int64_t seg_end = min(ct.t_e, split_run_end(plan, t));
            // Column sums of relu(K): each tile's 8 rows in plain binary32 pairs, folded into a
            // compensated binary32 running sum (sum + running error term) once per tile, in a
            // fixed order: FP64-class accuracy at FP32 rate.  Pair e holds columns
            // {4e, 4e + 2} (e < 2) or {4(e-2) + 1, 4(e-2) + 3} of the thread's chunk.
            uint64_t ks[4], kc[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) ks[e] = kc[e] = 0ull;
            for (; t < seg_end; ++t, ++it) {
                const uint32_t st = it % L::stages, ph = (it / L::stages) & 1u;
                const uint32_t tslot = it % L::tab_ring, tpar = (it / L::tab_ring) & 1u;
                // Every transform thread waits for both the K/V stage and the table slot (also
                // the threads with no columns to turn): the table ring is shorter than the K/V
                // ring, so only a thread that has seen a slot's rows land may free it again.
                if (!mbar_wait(full0 + 8u * st, ph, abort_flag, status, wait_ns) ||
                    !mbar_wait(tab_full0 + 8u * tslot, tpar, abort_flag, status, wait_ns)) {
                    ok = false;
                    break;
                }
                if (live) {
                    // Rows past the end of the sequence hold zeros in both the K and the table
                    // tiles (the copies fill outside the tensor with zeros): they rotate to zero
                    // and add zero to the sums, so every row is transformed without a test.
                    uint8_t* stage = base_ptr + st * L::stage_bytes;
                    uint8_t* atom = stage + (c >> 3) * kKvAtomBytes;
                    const uint8_t* tab = base_ptr + L::tab_offset + tslot * 2u * L::tab_bytes + 16 * c;  // [64][pairs]
                    uint64_t ts[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                    for (int k = 0; k < kKvTile / kGroups; ++k) {
                        const int r = rg + kGroups * k;
                        {
                            uint4* cell = reinterpret_cast<uint4*>(atom + r * 128 + (((c & 7) ^ (r & 7)) << 4));
                            uint4 w = *cell;
                            const float4 c4 = *reinterpret_cast<const float4*>(tab + r * pairs * 4);
                            const float4 s4 = *reinterpret_cast<const float4*>(tab + L::tab_bytes + r * pairs * 4);
                            uint64_t a0[2], a1[2];
                            rope_chunk(w, c4, s4, a0, a1);
                            ts[0] = f32x2_add(ts[0], a0[0]);
                            ts[1] = f32x2_add(ts[1], a0[1]);
                            ts[2] = f32x2_add(ts[2], a1[0]);
                            ts[3] = f32x2_add(ts[3], a1[1]);
                            *cell = w;
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint64_t yv = f32x2_sub(ts[e], kc[e]);
                        const uint64_t tsum = f32x2_add(ks[e], yv);
                        kc[e] = f32x2_sub(f32x2_sub(tsum, ks[e]), yv);
                        ks[e] = tsum;
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(tab_empty0 + 8u * tslot);
                mbar_arrive(ready0 + 8u * st);
            }
            if (!ok) break;
            // This row group's column sums of the segment: [h][slot][rg][column] (the
            // reduction adds the row groups in order, then the segments).
            if (live) {
                const int64_t slot = static_cast<int64_t>(h) * plan.seg_stride + segment_of(plan, h, ct.c);
                double* dst = pa.ksum_partial + (slot * kGroups + rg) * head_dim + 8 * c;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float s0, s1, c0, c1;
                    f32x2_unpack(ks[e], s0, s1);
                    f32x2_unpack(kc[e], c0, c1);
                    const int col = e < 2 ? 4 * e : 4 * (e - 2) + 1;
                    dst[col] = static_cast<double>(s0) - static_cast<double>(c0);
                    dst[col + 2] = static_cast<double>(s1) - static_cast<double>(c1);
                }
            }
        }
    } else if (!FUSED || warp < 6) {
        // ---------------- epilogue: TMEM lanes 32q..32q+31 = rows i of the partial KV.
        // Thread i keeps its row of the segment's running sum in registers (plain kernel) or in
        // TMEM columns sum_col.. (fused kernel); either way each finished sub-chunk is added into
        // it with one FP32 add per element, in sub-chunk order.
        const int q = warp & 3;
        const int i = 32 * q + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        uint32_t sub = 0;
        bool ok = true;
        for (int64_t t = ct.t_s; ok && t < ct.t_e;) {
            const int h = split_tile(plan, t).h;
            const int64_t seg_end = min(ct.t_e, split_run_end(plan, t));
            float acc[FUSED ? 1 : 64 * NBOX];
            if constexpr (!FUSED) {
#pragma unroll
                for (int c = 0; c < 64 * NBOX; ++c) acc[c] = 0.f;
            }
            for (int64_t k0 = t; k0 < seg_end; k0 += PROMOTE, ++sub) {
                const uint32_t buf = sub & 1u;
                if (!mbar_wait(acc_full0 + 8u * buf, (sub >> 1) & 1u, abort_flag, status, wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem + lane_base + buf * 128u;
#pragma unroll
                for (int c = 0; c < 4 * NBOX; ++c) {
                    if (16 * c < head_dim) {
                        uint32_t r[16];
                        tmem_ld16_sync(taddr + 16u * c, r);
                        if constexpr (FUSED) {
                            const uint32_t saddr = tmem + lane_base + L::sum_col + 16u * c;
                            uint32_t sv[16];
                            if (k0 == t) {
#pragma unroll
                                for (int e = 0; e < 16; ++e) sv[e] = __float_as_uint(__fadd_rn(0.f, __uint_as_float(r[e])));
                            } else {
                                tmem_ld16_sync(saddr, sv);
#pragma unroll
                                for (int e = 0; e < 16; ++e)
                                    sv[e] = __float_as_uint(__fadd_rn(__uint_as_float(sv[e]), __uint_as_float(r[e])));
                            }
                            tmem_st16(saddr, sv);
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e) acc[16 * c + e] += __uint_as_float(r[e]);
                        }
                    }
                }
                if constexpr (FUSED) tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty0 + 8u * buf);
            }
            if (!ok) break;
            const int64_t slot = static_cast<int64_t>(h) * plan.seg_stride + segment_of(plan, h, ct.c);
            float* dst = partial + (slot * head_dim + i) * head_dim;
#pragma unroll
            for (int c = 0; c < 4 * NBOX; ++c) {
                if (16 * c < head_dim) {
                    float v[16];
                    if constexpr (FUSED) {
                        uint32_t sv[16];
                        tmem_ld16_sync(tmem + lane_base + L::sum_col + 16u * c, sv);  // warp-collective
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(sv[e]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[e] = acc[16 * c + e];
                    }
                    if (i < head_dim) {
                        float4* o = reinterpret_cast<float4*>(dst + 16 * c);
#pragma unroll
                        for (int e = 0; e < 4; ++e) o[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                    }
                }
            }
            t = seg_end;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::tmem_cols);
    }
}

// ============================================================================ reduction
// kv[h][i][j] = the head's partials added in a fixed pairwise order: groups of 32 partials
// are each reduced as a tree (level w adds partial s + w into s for every s that is a
// multiple of 2w), then the group sums are reduced the same way.  The shape fixes the
// number of partials and so the order.
//
// The three-term BF16 image of KV^T is written in the apply MMA's B layout: row j,
// columns i = 8r .. 8r+7 form one 16-byte chunk in 64-column atom r / 8 of the
// 128-byte-swizzled K-major layout, at chunk position (r % 8) ^ (j % 8) of row j.
constexpr int kTreeGroup = 32;
constexpr int kTreeGroups = (kMaxSegments + kTreeGroup - 1) / kTreeGroup;

template <int N>
__device__ __forceinline__ float pairwise_sum(float (&v)[N], int count) {
#pragma unroll
    for (int w = 1; w < N; w *= 2) {
#pragma unroll
        for (int s = 0; s + w < N; s += 2 * w)
            if (s + w < count) v[s] = v[s] + v[s + w];
    }
    return v[0];
}

__device__ __forceinline__ float reduce_segments(const float* p, int64_t stride, int nseg) {
    float groups[kTreeGroups];
    int ngroups = 0;
#pragma unroll
    for (int g = 0; g < kTreeGroups; ++g) {
        const int g0 = g * kTreeGroup;
        if (g0 < nseg) {
            float vals[kTreeGroup];
#pragma unroll
            for (int s = 0; s < kTreeGroup; ++s) vals[s] = g0 + s < nseg ? p[(g0 + s) * stride] : 0.f;
            groups[g] = pairwise_sum(vals, nseg - g0);
            ngroups = g + 1;
        } else {
            groups[g] = 0.f;
        }
    }
    return pairwise_sum(groups, ngroups);
}

// Fixed-order sum of a head's FP64 column-sum partials (fused path): each segment's value
// is its row-group sums added in order (p[s][0..groups-1], `stride` apart), then the
// segments are added with the same tree as above.
__device__ __forceinline__ double segment_value_f64(const double* p, int64_t stride, int s, int groups) {
    const double* q = p + static_cast<int64_t>(s) * groups * stride;
    double v = q[0];
    for (int g = 1; g < groups; ++g) v += q[g * stride];
    return v;
}
// The same value with every load issued before the first add (one thread per segment).
__device__ __forceinline__ double segment_value_f64_wide(const double* p, int64_t stride, int s, int groups) {
    const double* q = p + static_cast<int64_t>(s) * groups * stride;
    double x[kKsumGroupsMax];
#pragma unroll
    for (int g = 0; g < kKsumGroupsMax; ++g) x[g] = g < groups ? q[g * stride] : 0.0;
    double v = x[0];
#pragma unroll
    for (int g = 1; g < kKsumGroupsMax; ++g)
        if (g < groups) v += x[g];
    return v;
}
__device__ __forceinline__ double reduce_segments_f64(const double* p, int64_t stride, int nseg, int row_groups) {
    double groups[kTreeGroups];
    int ngroups = 0;
#pragma unroll
    for (int g = 0; g < kTreeGroups; ++g) {
        const int g0 = g * kTreeGroup;
        groups[g] = 0.0;
        if (g0 < nseg) {
            double vals[kTreeGroup];
#pragma unroll
            for (int s = 0; s < kTreeGroup; ++s) vals[s] = g0 + s < nseg ? segment_value_f64(p, stride, g0 + s, row_groups) : 0.0;
#pragma unroll
            for (int w = 1; w < kTreeGroup; w *= 2)
#pragma unroll
                for (int s = 0; s + w < kTreeGroup; s += 2 * w)
                    if (s + w < nseg - g0) vals[s] = vals[s] + vals[s + w];
            groups[g] = vals[0];
            ngroups = g + 1;
        }
    }
#pragma unroll
    for (int w = 1; w < kTreeGroups; w *= 2)
#pragma unroll
        for (int s = 0; s + w < kTreeGroups; s += 2 * w)
            if (s + w < ngroups) groups[s] = groups[s] + groups[s + w];
    return groups[0];
}

// One CTA per 8-row slab of one head's KV (all D columns): thread (row e, column lane jl)
// takes the elements (8r + e, jl + 32 cb).  With at most kSmallSegs partials per head
// (every head count from 10 up) all of a thread's loads are issued before any add, so a
// slab costs one round trip to L2 and the reduction is a single wave of D/8 x H CTAs;
// with more partials each element goes through reduce_segments in turn.  The partials of
// an element are added in the same fixed pairwise order either way (pairwise_sum over 16
// values performs the same additions as over 32 when at most 16 are present).
constexpr int kSmallSegs = 16;
constexpr int kColBlocks = 4;  // 32-column blocks: head_dim <= 128

// The partials (and column-sum partials) are written by the kernel before this one in the
// stream, which may still be running when this grid starts: they are read through plain
// pointers, never `__restrict__` ones, so that no load of them can be treated as invariant
// and moved above the grid-dependency wait.
template <bool SMALL>
__global__ void __launch_bounds__(256, 2) kv_finalize_kernel(const float* partial, float* __restrict__ kv,
                                                             uint8_t* __restrict__ image, int h0, int head_dim,
                                                             const KvPlan plan, const double* ksum_partial,
                                                             float* __restrict__ ksum) {
    grid_launch_dependents();  // the apply kernel may start its prologue and Q loads now
    grid_dependency_wait();    // the partials of this call are complete past this point
    __shared__ float tile[kColBlocks][8][33];
    __shared__ double ks_seg[kSmallSegs][8];
    const int h = h0 + blockIdx.y;
    const int dd = head_dim * head_dim;
    const int r = blockIdx.x;  // rows 8r .. 8r+7
    const int e = threadIdx.x >> 5, jl = threadIdx.x & 31;
    const int i = 8 * r + e;
    const int ncb = (head_dim + 31) / 32;
    const int nseg = segments_of_head(plan, h);
    const float* p = partial + static_cast<int64_t>(h) * plan.seg_stride * dd + i * head_dim + jl;
    float* kv_row = kv + static_cast<int64_t>(h) * dd + i * head_dim + jl;
    if constexpr (SMALL) {
        float v[kColBlocks][kSmallSegs];
#pragma unroll
        for (int cb = 0; cb < kColBlocks; ++cb)
#pragma unroll
            for (int sg = 0; sg < kSmallSegs; ++sg)
                v[cb][sg] = (cb < ncb && jl + 32 * cb < head_dim && sg < nseg) ? p[sg * dd + 32 * cb] : 0.f;
#pragma unroll
        for (int cb = 0; cb < kColBlocks; ++cb) {
            const float x = pairwise_sum(v[cb], nseg);
            if (cb < ncb && jl + 32 * cb < head_dim) kv_row[32 * cb] = x;
            tile[cb][e][jl] = x;
        }
    } else {
#pragma unroll 1
        for (int cb = 0; cb < ncb; ++cb) {
            const float x = jl + 32 * cb < head_dim ? reduce_segments(p + 32 * cb, dd, nseg) : 0.f;
            if (jl + 32 * cb < head_dim) kv_row[32 * cb] = x;
            tile[cb][e][jl] = x;
        }
    }
    if (ksum_partial != nullptr) {
        // Fused path: the column sums of relu(K) of columns 8r .. 8r+7 over all tokens, each
        // segment's row groups in order, then the segments in the same tree; rounded once to FP32.
        const int groups = ksum_groups(head_dim);
        const double* kp = ksum_partial + static_cast<int64_t>(h) * plan.seg_stride * groups * head_dim;
        const int t = threadIdx.x;
        if constexpr (SMALL) {
            if (t < 8 * nseg) ks_seg[t >> 3][t & 7] = segment_value_f64_wide(kp + 8 * r + (t & 7), head_dim, t >> 3, groups);
            __syncthreads();
            if (t < 8) {
                double vals[kSmallSegs];
#pragma unroll
                for (int sg = 0; sg < kSmallSegs; ++sg) vals[sg] = sg < nseg ? ks_seg[sg][t] : 0.0;
#pragma unroll
                for (int w = 1; w < kSmallSegs; w *= 2)
#pragma unroll
                    for (int sg = 0; sg + w < kSmallSegs; sg += 2 * w)
                        if (sg + w < nseg) vals[sg] = vals[sg] + vals[sg + w];
                ksum[h * head_dim + 8 * r + t] = static_cast<float>(vals[0]);
            }
        } else if (t < 8) {
            ksum[h * head_dim + 8 * r + t] = static_cast<float>(reduce_segments_f64(kp + 8 * r + t, head_dim, nseg, groups));
        }
    }
    if (image == nullptr) return;
    __syncthreads();
    // The image: 32 threads per column block each write one 16-byte chunk (8 consecutive
    // rows i of column jj) per term.
    const int cb = threadIdx.x >> 5, jj = 32 * cb + jl;
    if (cb >= ncb || jj >= head_dim) return;
    uint32_t hi[4], mid[4], lo[4];
#pragma unroll
    for (int u = 0; u < 8; u += 2) {
        __nv_bfloat16 h2[2], m2[2], l2[2];
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            const float v = tile[cb][u + w][jl];
            h2[w] = __float2bfloat16_rn(v);
            const float r1 = v - __bfloat162float(h2[w]);  // exact
            m2[w] = __float2bfloat16_rn(r1);
            const float r2 = r1 - __bfloat162float(m2[w]);  // exact
            l2[w] = __float2bfloat16_rn(r2);
        }
        hi[u / 2] = static_cast<uint32_t>(__bfloat16_as_ushort(h2[0])) |
                    (static_cast<uint32_t>(__bfloat16_as_ushort(h2[1])) << 16);
        mid[u / 2] = static_cast<uint32_t>(__bfloat16_as_ushort(m2[0])) |
                     (static_cast<uint32_t>(__bfloat16_as_ushort(m2[1])) << 16);
        lo[u / 2] = static_cast<uint32_t>(__bfloat16_as_ushort(l2[0])) |
                    (static_cast<uint32_t>(__bfloat16_as_ushort(l2[1])) << 16);
    }
    const int atoms = head_dim_atoms(head_dim);
    const int64_t term_bytes = static_cast<int64_t>(atoms) * head_dim * 128;
    const int64_t off = static_cast<int64_t>(r >> 3) * head_dim * 128 + jj * 128 + (((r & 7) ^ (jj & 7)) << 4);
    uint8_t* img = image + static_cast<int64_t>(h) * 3 * term_bytes + off;
    *reinterpret_cast<uint4*>(img) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(img + term_bytes) = make_uint4(mid[0], mid[1], mid[2], mid[3]);
    *reinterpret_cast<uint4*>(img + 2 * term_bytes) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

template <int NBOX, bool FUSED, int PROMOTE>
cudaError_t launch_tc(const CUtensorMap& tm_k, const CUtensorMap& tm_v, float* partial, int head_dim,
                      const KvPlan& plan, const KvLaunch& work, bool token_major, int* status, uint64_t wait_ns,
                      cudaStream_t stream, const ProducerArgs& pa, const CUtensorMap& tm_cos,
                      const CUtensorMap& tm_sin) {
    using L = KvLayout<NBOX, FUSED>;
    cudaError_t e = cudaFuncSetAttribute(kv_partial_tc_kernel<NBOX, FUSED, PROMOTE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::smem_bytes);
    if (e != cudaSuccess) return e;
    return launch_overlapped(kv_partial_tc_kernel<NBOX, FUSED, PROMOTE>, dim3(work.n_chunks),
                             dim3(FUSED ? kKvThreadsFused : kKvThreads), L::smem_bytes, stream, tm_k, tm_v, partial,
                             head_dim, plan, work, token_major ? 1 : 0, status, wait_ns, pa, tm_cos, tm_sin);
}

}  // namespace

cudaError_t launch_kv_partial_tc(const CUtensorMap& tm_k, const CUtensorMap& tm_v, float* partial, int64_t n_tokens,
                                 int head_dim, const KvPlan& plan, const KvLaunch& work, bool token_major,
                                 bool lossless, int* status, uint64_t wait_ns, cudaStream_t stream,
                                 const ProducerArgs* producer, const CUtensorMap* tm_tables) {
    (void)n_tokens;
    const ProducerArgs pa = producer ? *producer : ProducerArgs{nullptr, nullptr, nullptr, nullptr, 0};
    const CUtensorMap none{};
    const CUtensorMap& tc = tm_tables ? tm_tables[0] : none;
    const CUtensorMap& ts = tm_tables ? tm_tables[1] : none;
    const bool one = head_dim_atoms(head_dim) == 1;
#define LA_KV_LAUNCH(NB, FU, PR) \
    launch_tc<NB, FU, PR>(tm_k, tm_v, partial, head_dim, plan, work, token_major, status, wait_ns, stream, pa, tc, ts)
    if (producer && lossless)
        return one ? LA_KV_LAUNCH(1, true, kPromoteLossless) : LA_KV_LAUNCH(2, true, kPromoteLossless);
    if (producer) return one ? LA_KV_LAUNCH(1, true, kPromoteHigh) : LA_KV_LAUNCH(2, true, kPromoteHigh);
    if (lossless) return one ? LA_KV_LAUNCH(1, false, kPromoteLossless) : LA_KV_LAUNCH(2, false, kPromoteLossless);
    return one ? LA_KV_LAUNCH(1, false, kPromoteHigh) : LA_KV_LAUNCH(2, false, kPromoteHigh);
#undef LA_KV_LAUNCH
}

cudaError_t launch_kv_finalize(const float* partial, float* kv, uint8_t* kv_image, int h0, int hc, int head_dim,
                               const KvPlan& plan, cudaStream_t stream, const ProducerArgs* producer) {
    dim3 grid(head_dim / 8, hc);
    const double* kp = producer ? producer->ksum_partial : nullptr;
    float* ks = producer ? producer->ksum : nullptr;
    if (plan.seg_stride <= kSmallSegs)
        return launch_overlapped(kv_finalize_kernel<true>, grid, dim3(256), 0, stream, partial, kv, kv_image, h0,
                                 head_dim, plan, kp, ks);
    return launch_overlapped(kv_finalize_kernel<false>, grid, dim3(256), 0, stream, partial, kv, kv_image, h0, head_dim,
                             plan, kp, ks);
}

}  // namespace la
