// Second GEMM + normalisation of the fused producer path, computed transposed:
//     out[h][n][j] = (sum_i Q_rot[h][n][i] KV[h][i][j]) / den[h][n]
//     as out^T = KV^T . Q_rot^T per 128-token tile (M = output feature j, N = token n)
//
// Activations may be head-major [1, H, N, D] or token-major [1, N, H, D] (the model's
// projection layout); only the tensor-map coordinates and the schedule differ.
//
// Page "PR #35728 完整报告 - [diffusion] Accelerate SANA-Video linear attention in
// quality=high", 关键源码片段: (scores @ query_rotate.float()) * normalizer, with the
// producer step of SanaVideoLinearAttention.forward (ReLU, interleaved RoPE, the normaliser
// from the un-rotated ReLU'd Q and the column sums of ReLU'd K) done here on the Q tile.
//
// The KV image (KV^T split into three BF16 terms hi + mid + lo, which carry 24 bits of KV,
// so every product is exact in FP32 and the result has FP32-class accuracy) lives in TMEM
// as the A operand of tcgen05.mma, which leaves shared memory to the streams: Q tiles, the
// rotation-table rows and the output staging.  Per CTA (persistent; one chunk of the body +
// tail split: k CTAs per head on the first B tiles of every head, cut at the same tiles,
// and the spare CTAs on the remaining tiles of all heads):
//   warp 0      TMA Q tiles (K-major, 128-byte swizzle: the B operand as loaded) and
//               bulk-copies each half tile's table rows into a three-slot ring;
//   warp 1      3 terms x D/16 K-steps of tcgen05.mma M=128 (features) N=128 (tokens) into
//               one of two TMEM accumulators;
//   warps 2..9  epilogue, a thread per output feature (two warps per TMEM lane quarter,
//               each with two of a tile's four 32-token chunks; at D <= 64 the features sit
//               in both halves of the lanes and each warp takes one chunk): on a head change
//               they copy the head's image rows into TMEM; per chunk they scale by the
//               tokens' reciprocal denominators and write [token][feature] boxes to staging
//               for TMA stores;
//   warps 10..25 producer step: ReLU + rotation of the Q tile in place, the row
//               normaliser, its correctly rounded reciprocal to the epilogue.
// The two warp groups that do per-element work are wide (8 and 16 warps) because each
// one's work per tile is a chain of dependent steps: more warps hide more latency.
#include <cuda_bf16.h>

#include "lin_attn_internal.cuh"
#include "ptx.cuh"

namespace la {
namespace {

constexpr int kFEpiWarps = 8;                       // warps 2..9
constexpr int kFXfWarps = 16;                       // warps 10..25
constexpr int kFXfWarp0 = 2 + kFEpiWarps;
constexpr int kFThreads = 32 * (kFXfWarp0 + kFXfWarps);
constexpr int kFTransformThreads = 32 * kFXfWarps;
constexpr int kFTabSubs = 2;                        // table slots per tile (half a tile of rows each)
constexpr int kFTabSlots = 3 * kFTabSubs / 2;       // table ring: 1.5 tiles of rows
constexpr uint32_t kFOutBufs = 1;                   // staging buffers per epilogue warp
// Reciprocal-denominator buffers between the transform and the epilogue.  A buffer is
// written by the transform of tile i and freed by the epilogue of tile i after the MMA, so
// the ring must span the whole transform -> MMA -> epilogue chain (~9000 cycles at
// D = 112, ~2 tile periods): with 2 buffers that chain, not any one stage, set the pace;
// 3 cover it (4 do not fit beside the D = 128 layout).
constexpr uint32_t kFDenBufs = 3;
constexpr int kFTabRows = kApplyTile / kFTabSubs;   // tokens per table slot
constexpr uint32_t kFQAtom = kApplyTile * 128;      // 128 token rows x 128 bytes
constexpr uint32_t kFBoxBytes = 32 * 128;           // staging box: 32 tokens x 128 bytes
constexpr uint32_t kFBarBytes = 512;
constexpr uint32_t kFSmemLimit = 232448;
constexpr uint32_t kFAccCols = 128;                 // one accumulator: 128 tokens
constexpr uint32_t kFImgCol = 2 * kFAccCols;        // image terms start after the two accumulators

__host__ __device__ constexpr int fused_stages(int nbox) { return nbox == 1 ? 6 : 3; }
__host__ __device__ constexpr uint32_t fused_tab_slot_bytes(int head_dim) {
    return static_cast<uint32_t>(kFTabRows) * (head_dim / 2) * 4u * 2u;
}
__host__ __device__ constexpr uint32_t fused_smem_bytes(int head_dim) {
    return fused_stages(head_dim_atoms(head_dim)) * head_dim_atoms(head_dim) * kFQAtom +
           kFTabSlots * fused_tab_slot_bytes(head_dim) + kFEpiWarps * kFOutBufs * kFBoxBytes + kFBarBytes +
           kFDenBufs * kApplyTile * 4 + 1024;
}
static_assert(fused_smem_bytes(128) <= kFSmemLimit && fused_smem_bytes(64) <= kFSmemLimit,
              "fused apply layout exceeds shared memory");
static_assert(kFImgCol + 3 * 64 <= 512, "accumulators and image exceed TMEM");
static_assert((3 * fused_stages(1) + 4 + 2 * kFDenBufs + 2 * kFTabSlots + 3) * 8 <= kFBarBytes - 64,
              "barriers overlap the TMEM address slot");

template <int NBOX, bool OUT_BF16>
__global__ void __launch_bounds__(kFThreads, 1)
    apply_fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_out,
                       const uint8_t* kv_image, int heads, int n_tokens, int head_dim,
                       const TileSplit sp, int token_major, int* status, uint64_t wait_ns,
                       const ProducerArgs pa) {
    constexpr int kStages = fused_stages(NBOX);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);

    const uint32_t tab_slot = fused_tab_slot_bytes(head_dim);
    const uint32_t q_smem = base;
    const uint32_t tab_smem = q_smem + kStages * NBOX * kFQAtom;
    const uint32_t o_smem = tab_smem + kFTabSlots * tab_slot;
    const uint32_t bar_off = o_smem + kFEpiWarps * kFOutBufs * kFBoxBytes - base;
    const uint32_t bars = base + bar_off;
    const uint32_t q_full0 = bars;                             // [stages] Q tile landed
    const uint32_t q_empty0 = q_full0 + 8u * kStages;          // [stages] its MMAs are done
    const uint32_t q_ready0 = q_empty0 + 8u * kStages;         // [stages] transformed
    const uint32_t acc_full0 = q_ready0 + 8u * kStages;        // [2]
    const uint32_t acc_empty0 = acc_full0 + 16u;               // [2]
    const uint32_t den_full0 = acc_empty0 + 16u;               // [kFDenBufs] reciprocal denominators written
    const uint32_t den_empty0 = den_full0 + 8u * kFDenBufs;    // [kFDenBufs] ... and read
    const uint32_t tab_full0 = den_empty0 + 8u * kFDenBufs;    // [kFTabSlots]
    const uint32_t tab_empty0 = tab_full0 + 8u * kFTabSlots;   // [kFTabSlots]
    const uint32_t b_full = tab_empty0 + 8u * kFTabSlots;      // the head's image is in TMEM
    const uint32_t b_empty = b_full + 8u;                      // the old image's MMAs are done
    const uint32_t drain_bar = b_empty + 8u;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + bar_off + kFBarBytes - 64);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + bar_off + kFBarBytes - 56);
    float* rcp_s = reinterpret_cast<float*>(base_ptr + bar_off + kFBarBytes);  // [kFDenBufs][kApplyTile]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // The CTAs are the chunks of the body + tail split sp: k CTAs per head take the first
    // B tiles of their head, cut at the same tiles for every head, so the CTAs running
    // together work on the same token rows.  They then read each rotation-table row (the
    // same for every head) from DRAM once, and token-major activations on whole DRAM rows.
    // The 152 - k H spare CTAs share the remaining tiles of all heads (a few MB of tables,
    // which stay in L2).  (Contiguous ranges of the (head, tile) sequence keep all SMs busy
    // too, but the CTAs then walk the whole token range at once and the 80 MB of tables at
    // 720p were read from DRAM about five times: 0.8 % slower per call.)
    const int t_begin = static_cast<int>(split_begin(sp, blockIdx.x));
    const int t_end = static_cast<int>(split_begin(sp, blockIdx.x + 1));
    const uint32_t half_d = static_cast<uint32_t>(head_dim / 2);  // image columns per term

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(q_full0 + 8u * s, 1);
            mbar_init(q_empty0 + 8u * s, 1);
            mbar_init(q_ready0 + 8u * s, kFTransformThreads);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full0 + 8u * b, 1);
            mbar_init(acc_empty0 + 8u * b, kFEpiWarps);
        }
        for (uint32_t b = 0; b < kFDenBufs; ++b) {
            mbar_init(den_full0 + 8u * b, kFTransformThreads);
            mbar_init(den_empty0 + 8u * b, kFEpiWarps);
        }
        for (int s = 0; s < kFTabSlots; ++s) {
            mbar_init(tab_full0 + 8u * s, 1);
            mbar_init(tab_empty0 + 8u * s, kFTransformThreads);
        }
        mbar_init(b_full, kFEpiWarps);
        mbar_init(b_empty, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), 512);
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
    grid_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- producer: Q tiles (inputs of the call) and table rows
            // Token-major Q rows share DRAM granules with the neighbouring heads' rows, which
            // other CTAs read at about the same time: those lines stay at normal priority.
            const uint64_t pol = token_major ? policy_evict_normal() : policy_evict_first();
            const uint64_t tpol = policy_evict_last();  // every head of the layer re-reads the tables
            const uint32_t row_bytes = half_d * 4u;
            uint32_t q_issued = 0, tab_issued = 0;  // copies issued (for the wind-down)
            bool ok = true;
            for (int t = t_begin; t < t_end && ok; ++t) {
                const uint32_t it = static_cast<uint32_t>(t - t_begin);
                int h, tile;
                split_tile32(sp, t, h, tile);
                const int n0 = tile * kApplyTile;
                const uint32_t st = it % kStages, ph = (it / kStages) & 1u;
                if (!(ok = mbar_wait(q_empty0 + 8u * st, ph ^ 1u, abort_flag, status, wait_ns))) break;
                mbar_arrive_expect_tx(q_full0 + 8u * st, NBOX * kFQAtom);
#pragma unroll
                for (int x = 0; x < NBOX; ++x)
                    tma_load_3d_hint(q_smem + (st * NBOX + x) * kFQAtom, &tm_q, q_full0 + 8u * st, 64 * x,
                                     token_major ? h : n0, token_major ? n0 : h, pol);
                q_issued = it + 1;
                // The tile's rotation-table rows, half a tile per slot: rows of the [N][D/2]
                // tables are contiguous, so a slot is one bulk copy per table, cut at N.
                for (uint32_t hh = 0; hh < kFTabSubs && ok; ++hh) {
                    const uint32_t i = kFTabSubs * it + hh;
                    const uint32_t slot = i % kFTabSlots, tph = (i / kFTabSlots) & 1u;
                    if (!(ok = mbar_wait(tab_empty0 + 8u * slot, tph ^ 1u, abort_flag, status, wait_ns))) break;
                    const int r0 = n0 + static_cast<int>(hh) * kFTabRows;
                    const int rows = max(0, min(kFTabRows, n_tokens - r0));
                    const uint32_t bytes = static_cast<uint32_t>(rows) * row_bytes;
                    const uint32_t dst = tab_smem + slot * tab_slot;
                    mbar_arrive_expect_tx(tab_full0 + 8u * slot, 2u * bytes);
                    if (rows > 0) {
                        bulk_load_hint(dst, pa.cos + static_cast<int64_t>(r0) * half_d, bytes, tab_full0 + 8u * slot,
                                       tpol);
                        bulk_load_hint(dst + tab_slot / 2, pa.sin + static_cast<int64_t>(r0) * half_d, bytes,
                                       tab_full0 + 8u * slot, tpol);
                    }
                    tab_issued = i + 1;
                }
            }
            // Let the copies in flight land before the CTA exits: the consumers wait for all of
            // them unless some role gave up, in which case nothing else would.
            const uint32_t first = q_issued > kStages ? q_issued - kStages : 0;
            for (uint32_t j = first; j < q_issued; ++j)
                mbar_wait_drain(q_full0 + 8u * (j % kStages), (j / kStages) & 1u);
            const uint32_t tfirst = tab_issued > kFTabSlots ? tab_issued - kFTabSlots : 0u;
            for (uint32_t j = tfirst; j < tab_issued; ++j)
                mbar_wait_drain(tab_full0 + 8u * (j % kFTabSlots), (j / kFTabSlots) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer: out^T (features x tokens) += KV^T term x Q^T
            const uint32_t idesc = make_idesc_bf16_f32(128, kApplyTile, false, false);
            const int ksteps = head_dim / 16;
            uint32_t it = 0;
            int cur_h = -1, run = -1;
            for (int t = t_begin; t < t_end; ++t, ++it) {
                int h, tile;
                split_tile32(sp, t, h, tile);
                const uint32_t lt = static_cast<uint32_t>(t - t_begin);
                if (h != cur_h) {
                    if (run >= 0) mma_commit(b_empty);  // the old image is free once its MMAs are done
                    ++run;
                    cur_h = h;
                    if (!mbar_wait(b_full, run & 1, abort_flag, status, wait_ns)) break;
                    tc_fence_after();
                }
                const uint32_t buf = lt & 1u;
                if (!mbar_wait(acc_empty0 + 8u * buf, ((lt >> 1) & 1u) ^ 1u, abort_flag, status, wait_ns)) break;
                const uint32_t st = it % kStages, ph = (it / kStages) & 1u;
                if (!mbar_wait(q_ready0 + 8u * st, ph, abort_flag, status, wait_ns)) break;
                tc_fence_after();
                const uint32_t d = tmem + buf * kFAccCols;
                const uint32_t qb = q_smem + st * NBOX * kFQAtom;
                // Smallest term first; every product is exact, the accumulator is FP32.
#pragma unroll
                for (int term = 2; term >= 0; --term) {
                    for (int ks = 0; ks < ksteps; ++ks) {
                        const uint32_t off = (ks >> 2) * kFQAtom + (ks & 3) * 32u;
                        mma_bf16_ts(d, tmem + kFImgCol + term * half_d + 8u * ks,
                                    make_smem_desc(qb + off, 16u, 1024u, kSwizzle128B), idesc,
                                    (term != 2 || ks != 0) ? 1u : 0u);
                    }
                }
                mma_commit(q_empty0 + 8u * st);
                mma_commit(acc_full0 + 8u * buf);
            }
            mma_commit(drain_bar);
            mbar_wait_drain(drain_bar, 0);
        }
    } else if (warp >= kFXfWarp0) {
        // ---------------- producer-step transform of the Q tiles
        // Thread (chunk c, row group rg) takes columns 8c..8c+7 of rows rg + G k, with
        // kCpr = 16 chunk lanes per row and G = 32 row groups (4 rows a thread) when the head
        // dim spans two 64-column atoms, 8 lanes and 64 groups (2 rows) when it fits one:
        // ReLU, dot with the head's column sums of relu(K) (the normaliser), then the rotation
        // (binary32 products and sum in a fixed order, rounded once to BF16).  The threads of
        // a row add their dot products in a fixed butterfly; the row's reciprocal denominator
        // (correctly rounded) goes to rcp_s for the epilogue.
        constexpr int kCpr = 8 * NBOX;                   // chunk lanes per row
        constexpr int kRowGroups = kFTransformThreads / kCpr;
        static_assert(kFTabRows % kRowGroups == 0, "a table slot must hold whole row groups");
        const int u = threadIdx.x - 32 * kFXfWarp0;
        const int c = u % kCpr, rg = u / kCpr;
        const bool live = 8 * c < head_dim;
        const uint32_t row_bytes = half_d * 4u;
        uint64_t ks[4];  // the head's column sums in rope_chunk's activation order
        int cur_h = -1;
        uint32_t it = 0;
        for (int t = t_begin; t < t_end; ++t, ++it) {
            int h, tile;
            split_tile32(sp, t, h, tile);
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
            const uint32_t st = it % kStages, ph = (it / kStages) & 1u;
            const uint32_t db = lt % kFDenBufs, dph = (lt / kFDenBufs) & 1u;
            if (!mbar_wait(q_full0 + 8u * st, ph, abort_flag, status, wait_ns)) break;
            if (!mbar_wait(den_empty0 + 8u * db, dph ^ 1u, abort_flag, status, wait_ns)) break;
            uint8_t* atom = base_ptr + (q_smem - base) + (st * NBOX + (c >> 3)) * kFQAtom;
            bool ok = true;
#pragma unroll
            for (int hh = 0; hh < kFTabSubs; ++hh) {
                const uint32_t i = kFTabSubs * it + hh;
                const uint32_t slot = i % kFTabSlots;
                if (!(ok = mbar_wait(tab_full0 + 8u * slot, (i / kFTabSlots) & 1u, abort_flag, status, wait_ns))) break;
                const uint8_t* tab = base_ptr + (tab_smem - base) + slot * tab_slot + 16 * c;
                constexpr int kPer = kFTabRows / kRowGroups;  // this thread's rows per slot
                float part[kPer];
                if (live) {
                    // All of the slot's loads first, then the arithmetic: the rows' chains overlap.
                    // Rows past the end of the sequence are not tested for: their Q is zero (the
                    // copy fills outside the tensor with zeros), so their normaliser is the
                    // constant; their table rows were not copied, so what they compute is never
                    // used - an output column depends on its own token's row only, and the
                    // stores stop at N.
                    uint4* cell[kPer];
                    uint4 w[kPer];
                    float4 c4[kPer], s4[kPer];
#pragma unroll
                    for (int kk = 0; kk < kPer; ++kk) {
                        const int r = rg + kRowGroups * (kPer * hh + kk);
                        const uint32_t tr = static_cast<uint32_t>(r - hh * kFTabRows) * row_bytes;
                        cell[kk] = reinterpret_cast<uint4*>(atom + r * 128 + (((c & 7) ^ (r & 7)) << 4));
                        w[kk] = *cell[kk];
                        c4[kk] = *reinterpret_cast<const float4*>(tab + tr);
                        s4[kk] = *reinterpret_cast<const float4*>(tab + tab_slot / 2 + tr);
                    }
#pragma unroll
                    for (int kk = 0; kk < kPer; ++kk) {
                        uint64_t a0[2], a1[2];
                        rope_chunk(w[kk], c4[kk], s4[kk], a0, a1);
                        uint64_t d2 = f32x2_mul(a0[0], ks[0]);
                        d2 = f32x2_fma(a0[1], ks[1], d2);
                        d2 = f32x2_fma(a1[0], ks[2], d2);
                        d2 = f32x2_fma(a1[1], ks[3], d2);
                        float d0, d1;
                        f32x2_unpack(d2, d0, d1);
                        part[kk] = d0 + d1;
                        *cell[kk] = w[kk];
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < kPer; ++kk) part[kk] = 0.f;
                }
#pragma unroll
                for (int kk = 0; kk < kPer; ++kk) {
                    const int r = rg + kRowGroups * (kPer * hh + kk);
                    float p = part[kk];
#pragma unroll
                    for (int m = kCpr / 2; m >= 1; m >>= 1) p += __shfl_xor_sync(0xffffffffu, p, m);
                    if (c == 0) rcp_s[db * kApplyTile + r] = __frcp_rn(p + kDenEps);
                }
                mbar_arrive(tab_empty0 + 8u * slot);
            }
            if (!ok) break;
            fence_proxy_async_smem();
            mbar_arrive(q_ready0 + 8u * st);
            mbar_arrive(den_full0 + 8u * db);
        }
    } else {
        // ---------------- epilogue: warp (q = warp % 4) owns TMEM lanes 32q..32q+31, thread =
        // output feature j.  When the head dim spans two atoms, lane = feature and half e takes
        // token chunks 2e, 2e + 1 of each tile.  When it fits one (D <= 64), lanes 64..127 hold
        // a second copy of features 0..63 (the image rows are written twice, so the product
        // computes them twice at no cost: M is 128 either way), and each of the eight warps
        // takes one chunk of one feature half - chunk 2e + q / 2, features 32 (q % 2) ... - so
        // that no warp sits idle on the empty upper lanes.
        const int q = warp & 3;
        const int e = (warp - 2) >> 2;
        const int j = NBOX == 1 ? 32 * (q & 1) + lane : 32 * q + lane;  // output feature
        const int fq = NBOX == 1 ? (q & 1) : q;                          // its 32-feature block
        const bool live = 32 * fq < head_dim;  // any of the warp's features exists
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const uint32_t stage0 = o_smem + static_cast<uint32_t>(warp - 2) * kFOutBufs * kFBoxBytes;
        // Token-major output rows share L2 lines with the neighbouring heads' rows (written by
        // other CTAs): normal priority, as for the loads.
        const uint64_t spol = token_major ? policy_evict_normal() : policy_evict_first();
        const int64_t term_bytes = static_cast<int64_t>(NBOX) * head_dim * 128;
        uint32_t nstore = 0;
        int cur_h = -1, run = -1;
        bool ok = true;
        for (int t = t_begin; t < t_end && ok; ++t) {
            int h, tile;
            split_tile32(sp, t, h, tile);
            const int n0 = tile * kApplyTile;
            const uint32_t lt = static_cast<uint32_t>(t - t_begin);
            if (h != cur_h) {
                // The head's image into TMEM: feature j's row of each term (input features i as
                // BF16 pairs), read from the swizzled image the reduction wrote.
                if (cur_h < 0) grid_dependency_wait();
                ++run;
                cur_h = h;
                if (run > 0 && !(ok = mbar_wait(b_empty, (run - 1) & 1, abort_flag, status, wait_ns))) break;
                tc_fence_after();
                const uint8_t* img = kv_image + static_cast<int64_t>(h) * 3 * term_bytes;
                const uint32_t groups = 3u * half_d / 8u;  // 8-word groups of the three terms
                for (uint32_t gi = e * ((groups + 1) / 2); gi < min(groups, (e + 1) * ((groups + 1) / 2)); ++gi) {
                    const uint32_t term = gi / (half_d / 8u), w0 = 8u * (gi % (half_d / 8u));
                    {  // 8 words = input features 2 w0 .. 2 w0 + 15
                        uint32_t wv[8];
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const uint32_t w = w0 + 4 * hf;            // first word of a 16-byte chunk
                            const uint32_t x = w >> 5, cc = (w & 31) >> 2;
                            uint4 v4 = make_uint4(0u, 0u, 0u, 0u);
                            if (j < head_dim)
                                v4 = *reinterpret_cast<const uint4*>(
                                    img + term * term_bytes + static_cast<int64_t>(x) * head_dim * 128 + j * 128 +
                                    ((cc ^ (static_cast<uint32_t>(j) & 7u)) << 4));
                            wv[4 * hf] = v4.x;
                            wv[4 * hf + 1] = v4.y;
                            wv[4 * hf + 2] = v4.z;
                            wv[4 * hf + 3] = v4.w;
                        }
                        tmem_st8(tmem + lane_base + kFImgCol + term * half_d + w0, wv);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(b_full);
            }
            const uint32_t buf = lt & 1u;
            const uint32_t db = lt % kFDenBufs, dph = (lt / kFDenBufs) & 1u;
            if (!(ok = mbar_wait(den_full0 + 8u * db, dph, abort_flag, status, wait_ns))) break;
            if (!(ok = mbar_wait(acc_full0 + 8u * buf, (lt >> 1) & 1u, abort_flag, status, wait_ns))) break;
            tc_fence_after();
            const float* rcp_t = rcp_s + db * kApplyTile;
            const int g0 = NBOX == 1 ? 2 * e + (q >> 1) : 2 * e, g1 = NBOX == 1 ? g0 + 1 : g0 + 2;
            for (int g = g0; g < g1 && n0 + 32 * g < n_tokens; ++g) {
                uint32_t r[32];
                tmem_ld32_sync(tmem + lane_base + buf * kFAccCols + 32u * g, r);
                if (!live) continue;
                const uint32_t sbuf = stage0 + (nstore % kFOutBufs) * kFBoxBytes;
                if (lane == 0) bulk_wait_read<kFOutBufs - 1>();
                __syncwarp();
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    const float4 rc = *reinterpret_cast<const float4*>(rcp_t + 32 * g + 4 * e4);
                    const float sc[4] = {rc.x, rc.y, rc.z, rc.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int tok = 4 * e4 + e;
                        const float v = __uint_as_float(r[tok]) * sc[e];
                        if (OUT_BF16) {
                            const uint16_t b = __bfloat16_as_ushort(__float2bfloat16_rn(v));
                            asm volatile("st.shared.b16 [%0], %1;" ::"r"(sbuf + tok * 64u + lane * 2u), "h"(b)
                                         : "memory");
                        } else {
                            asm volatile("st.shared.f32 [%0], %1;" ::"r"(sbuf + tok * 128u + lane * 4u), "f"(v)
                                         : "memory");
                        }
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d_hint(&tm_out, sbuf, 32 * fq, token_major ? h : n0 + 32 * g,
                                      token_major ? n0 + 32 * g : h, spol);
                    bulk_commit();
                }
                ++nstore;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(den_empty0 + 8u * db);
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
        tmem_dealloc(tmem, 512);
    }
}

template <int NBOX, bool BF16>
cudaError_t launch(const CUtensorMap& tm_q, const CUtensorMap& tm_out, const uint8_t* img, int heads, int n_tokens,
                   int head_dim, bool token_major, const TileSplit& sp, int* status, uint64_t wait_ns,
                   cudaStream_t stream, const ProducerArgs& pa) {
    const uint32_t smem = fused_smem_bytes(head_dim);
    cudaError_t e = cudaFuncSetAttribute(apply_fused_kernel<NBOX, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_overlapped(apply_fused_kernel<NBOX, BF16>, dim3(sp.chunks), dim3(kFThreads), smem, stream, tm_q,
                             tm_out, img, heads, n_tokens, head_dim, sp, token_major ? 1 : 0, status, wait_ns, pa);
}

}  // namespace

cudaError_t launch_apply_fused_tc(const CUtensorMap& tm_q, const CUtensorMap& tm_out_t, const uint8_t* kv_image,
                                  int heads, int64_t n_tokens, int head_dim, bool out_bf16, bool token_major, int grid,
                                  int* status, uint64_t wait_ns, cudaStream_t stream, const ProducerArgs& producer) {
    const int n = static_cast<int>(n_tokens);
    const int tph = (n + kApplyTile - 1) / kApplyTile;
    const TileSplit sp = tile_split(heads, tph, grid, kNoPerHeadCap, kApplyMinPart, kApplySwitchCost);  // a CTA per chunk
#define LA_FUSED(NB, BF) \
    launch<NB, BF>(tm_q, tm_out_t, kv_image, heads, n, head_dim, token_major, sp, status, wait_ns, stream, producer)
    if (head_dim_atoms(head_dim) == 1) return out_bf16 ? LA_FUSED(1, true) : LA_FUSED(1, false);
    return out_bf16 ? LA_FUSED(2, true) : LA_FUSED(2, false);
#undef LA_FUSED
}

}  // namespace la
