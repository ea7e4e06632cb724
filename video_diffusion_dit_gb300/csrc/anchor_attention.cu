// SANA-Video 2.0 softmax anchor attention on tensor cores (flash-attention forward).
//
// Page "[sglang] SANA-Video 2.0 anchor attention의 FP32 upcast 제거로 720p 생성 52%
// 단축하기" (PR #49219), section 코드 분석, 2. GatedSoftmaxAttention: the anchor layer is
// F.scaled_dot_product_attention(q, k, v, dropout_p=0.0) on BF16 [B, H, N, D] tensors (no
// mask, default scale 1/sqrt(D)); the page's 'high' tier hands BF16 Q/K/V to a flash
// kernel.  Here, per head, for two 128-query tiles t = 0, 1 at once:
//     S_t = Q_t K^T (tcgen05, FP32 in TMEM), P_t = exp2(S_t * scale * log2 e - m) (BF16,
//     written back over the upper half of S_t in TMEM), O_t += P_t V (tcgen05 with A read
//     from TMEM, FP32 in TMEM), out = O_t / sum(P_t)
// with the running maximum m kept per row and O rescaled only when a row's maximum grows
// by more than 8 (in log2 units) - the weights stay below 2^8, and O / sum(P) is exact for
// any reference m - so the rescale (a TMEM read-modify-write) is rare.
//
// The two query tiles ping-pong: while one softmax warpgroup turns S_t(j) into weights, the
// tensor pipe runs the other tile's products, in the issue order
//     PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), ...
// Tensor-core operations of one thread complete in issue order, so S_t(j) landing means
// PV_t(j-1) has landed too: the softmax warps may rescale O_t right then, and S_t(j+1) may
// overwrite the TMEM columns that PV_t(j) reads P_t(j) from.
#include <cuda_bf16.h>

#include "lin_attn_internal.cuh"
#include "ptx.cuh"

namespace la {
namespace {

constexpr int kBM = 128;                            // query rows per Q tile (MMA M, one row per thread)
constexpr int kQTiles = 2;                          // Q tiles per CTA, one softmax warpgroup each
constexpr int kBN = 128;                            // keys per K/V tile
constexpr int kSlots = 5;                           // K/V ring: each slot holds one K or one V tile
constexpr int kSoftmaxWarps = 4 * kQTiles;          // warps 0..7: softmax + epilogue
constexpr int kMmaWarp = kSoftmaxWarps;             // warp 8: TMEM owner and MMA issuer
constexpr int kTmaWarp = kSoftmaxWarps + 1;         // warp 9: TMA producer
constexpr int kAttnThreads = 32 * (kSoftmaxWarps + 2);
constexpr uint32_t kAtom = 128 * 128;               // 16 KB: 128 rows x 64 BF16 columns, 128-byte swizzle
constexpr float kRescaleSlack = 8.0f;               // rescale O when a row maximum grows by more than this
// TMEM columns: S_t at 128 t, P_t over S_t's columns 64..127, O_t at 256 + 128 t.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 256;
constexpr uint32_t kPCol = 64;

template <int NBOX>
struct AttnLayout {
    static constexpr uint32_t tile_bytes = NBOX * kAtom;  // one Q, K or V tile
    static constexpr uint32_t ring_offset = kQTiles * tile_bytes;
    static constexpr uint32_t bar_offset = ring_offset + kSlots * tile_bytes;
    static constexpr uint32_t smem_bytes = bar_offset + 256 + 1024;
};

// Weights of 64 keys of one row, p = 2^(s * scale_log2 - m), written as packed BF16 pairs
// (key 2c in the low half of column c) to the TMEM row at p_addr, 16 columns at a time;
// returns the sum of the unrounded weights (two paired partial sums, added in a fixed
// order).  The caller waits for the stores.
__device__ __forceinline__ float half_weights(const uint32_t (&s)[64], uint64_t scale2, uint64_t neg_m2,
                                              uint32_t p_addr) {
    uint64_t acc[2] = {0ull, 0ull};
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int c = 16 * g + i;
            float x0, x1;
            f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), scale2,
                                   neg_m2),
                         x0, x1);
            const float p0 = exp2_approx(x0), p1 = exp2_approx(x1);
            acc[c & 1] = f32x2_add(acc[c & 1], f32x2_pack(p0, p1));
            const __nv_bfloat162 pp = __floats2bfloat162_rn(p0, p1);
            pk[i] = *reinterpret_cast<const uint32_t*>(&pp);
        }
        tmem_st16(p_addr + 16u * g, pk);
    }
    float a0, a1, b0, b1;
    f32x2_unpack(acc[0], a0, a1);
    f32x2_unpack(acc[1], b0, b1);
    return (a0 + a1) + (b0 + b1);
}

template <int NBOX, bool OUT_BF16>
__global__ void __launch_bounds__(kAttnThreads, 1)
    anchor_attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, void* __restrict__ out, int n_tokens,
                            int head_dim, float scale_log2, int* status, uint64_t wait_ns) {
    using L = AttnLayout<NBOX>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);

    const uint32_t bars = base + L::bar_offset;
    const uint32_t q_full = bars;
    const uint32_t kv_full0 = bars + 8u;                      // [slots]
    const uint32_t kv_empty0 = kv_full0 + 8u * kSlots;        // [slots]
    const uint32_t s_full0 = kv_empty0 + 8u * kSlots;         // [tiles] S_t(j) in TMEM
    const uint32_t p_full0 = s_full0 + 8u * kQTiles;          // [tiles] P_t(j) in TMEM, O_t rescaled
    const uint32_t o_done = p_full0 + 8u * kQTiles;           // every product has landed
    const uint32_t drain_bar = o_done + 8u;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + L::bar_offset + 192);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + L::bar_offset + 200);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int q_blocks = (n_tokens + kQTiles * kBM - 1) / (kQTiles * kBM);
    const int h = blockIdx.x / q_blocks;
    const int m0 = (blockIdx.x % q_blocks) * (kQTiles * kBM);
    const int n_kv = (n_tokens + kBN - 1) / kBN;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(kv_full0 + 8u * s, 1);
            mbar_init(kv_empty0 + 8u * s, 1);
        }
        for (int t = 0; t < kQTiles; ++t) {
            mbar_init(s_full0 + 8u * t, 1);
            mbar_init(p_full0 + 8u * t, 4 * 32);
        }
        mbar_init(o_done, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_holder), kTmemCols);
        tmem_relinquish();
    }
    if (warp == kTmaWarp && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    auto slot_addr = [&](uint32_t i) { return base + L::ring_offset + (i % kSlots) * L::tile_bytes; };

    if (warp == kTmaWarp) {
        if (lane == 0) {
            // ---------------- producer: both Q tiles once, then K(0), V(0), K(1), V(1), ...
            const uint64_t pol_q = policy_evict_first();
            mbar_arrive_expect_tx(q_full, kQTiles * L::tile_bytes);
#pragma unroll
            for (int t = 0; t < kQTiles; ++t)
#pragma unroll
                for (int x = 0; x < NBOX; ++x)
                    tma_load_3d_hint(base + t * L::tile_bytes + x * kAtom, &tm_q, q_full, 64 * x, m0 + kBM * t, h,
                                     pol_q);
            const uint32_t n_loads = 2u * static_cast<uint32_t>(n_kv);
            uint32_t i = 0;
            for (; i < n_loads; ++i) {
                const uint32_t st = i % kSlots, ph = (i / kSlots) & 1u;
                if (!mbar_wait(kv_empty0 + 8u * st, ph ^ 1u, abort_flag, status, wait_ns)) break;
                mbar_arrive_expect_tx(kv_full0 + 8u * st, L::tile_bytes);
                const CUtensorMap* map = (i & 1u) ? &tm_v : &tm_k;
                const int key0 = static_cast<int>(i >> 1) * kBN;
#pragma unroll
                for (int x = 0; x < NBOX; ++x)
                    tma_load_3d(slot_addr(i) + x * kAtom, map, kv_full0 + 8u * st, 64 * x, key0, h);
            }
            // Let the copies in flight land before the CTA exits: the MMA issuer waits for all
            // of them unless some role gave up, in which case nothing else would.
            const uint32_t first = i > kSlots ? i - kSlots : 0;
            for (uint32_t k = first; k < i; ++k) mbar_wait_drain(kv_full0 + 8u * (k % kSlots), (k / kSlots) & 1u);
            mbar_wait_drain(q_full, 0);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            // ---------------- MMA issuer
            const uint32_t idesc_s = make_idesc_bf16_f32(kBM, kBN, false, false);      // Q, K both K-major
            const uint32_t idesc_o = make_idesc_bf16_f32(kBM, head_dim, false, true);  // P K-major (TMEM), V MN-major
            const int ksteps = head_dim / 16;
            auto wait_full = [&](uint32_t i) {
                return mbar_wait(kv_full0 + 8u * (i % kSlots), (i / kSlots) & 1u, abort_flag, status, wait_ns);
            };
            // Descriptors are built once per tile and advanced by the K-step's offset (the
            // start-address field is bits 0..13 of the descriptor, address >> 4, and no shared
            // address here carries out of it): the issuing thread, not the tensor pipe, had
            // been the limit with a descriptor built per instruction.
            const uint64_t q_desc[kQTiles] = {make_smem_desc(base, 16u, 1024u, kSwizzle128B),
                                              make_smem_desc(base + L::tile_bytes, 16u, 1024u, kSwizzle128B)};
            auto issue_s = [&](int t, uint32_t kslot) {
                const uint64_t kd = make_smem_desc(kslot, 16u, 1024u, kSwizzle128B);
#pragma unroll
                for (int ks = 0; ks < 4 * NBOX; ++ks) {
                    if (ks < ksteps) {
                        const uint64_t off = ((ks >> 2) * kAtom + (ks & 3) * 32u) >> 4;
                        mma_bf16(tmem + 128u * t, q_desc[t] + off, kd + off, idesc_s, ks != 0 ? 1u : 0u);
                    }
                }
                mma_commit(s_full0 + 8u * t);
            };
            auto issue_pv = [&](int t, uint32_t vslot, bool accumulate) {
                const uint64_t vd = make_smem_desc(vslot, kAtom, 1024u, kSwizzle128B);
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_bf16_ts(tmem + kOCol + 128u * t, tmem + 128u * t + kPCol + 8u * kk, vd + kk * (2048u >> 4),
                                idesc_o, (accumulate || kk != 0) ? 1u : 0u);
            };
            bool ok = mbar_wait(q_full, 0, abort_flag, status, wait_ns) && wait_full(0);
            if (ok) {
                tc_fence_after();
                issue_s(0, slot_addr(0));
                issue_s(1, slot_addr(0));
                mma_commit(kv_empty0 + 8u * (0 % kSlots));
            }
            for (uint32_t j = 0; ok && j < static_cast<uint32_t>(n_kv); ++j) {
                const uint32_t iv = 2 * j + 1, ik = 2 * j + 2;
                const bool more = j + 1 < static_cast<uint32_t>(n_kv);
                if (!(ok = wait_full(iv) && mbar_wait(p_full0, j & 1u, abort_flag, status, wait_ns))) break;
                tc_fence_after();
                issue_pv(0, slot_addr(iv), j > 0);
                if (more) {
                    if (!(ok = wait_full(ik))) break;
                    tc_fence_after();
                    issue_s(0, slot_addr(ik));
                }
                if (!(ok = mbar_wait(p_full0 + 8u, j & 1u, abort_flag, status, wait_ns))) break;
                tc_fence_after();
                issue_pv(1, slot_addr(iv), j > 0);
                mma_commit(kv_empty0 + 8u * (iv % kSlots));
                if (more) {
                    issue_s(1, slot_addr(ik));
                    mma_commit(kv_empty0 + 8u * (ik % kSlots));
                }
            }
            if (ok) mma_commit(o_done);
            mma_commit(drain_bar);
            mbar_wait_drain(drain_bar, 0);
        }
    } else {
        // ---------------- softmax and epilogue: warpgroup t, thread = query row r of Q tile t
        const int t = warp >> 2;
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const uint32_t s_addr = tmem + lane_base + 128u * t;
        const uint32_t o_addr = tmem + lane_base + kOCol + 128u * t;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            if (!(ok = mbar_wait(s_full0 + 8u * t, j & 1u, abort_flag, status, wait_ns))) break;
            tc_fence_after();
            // The whole row of S_t(j); keys past the end are masked out.
            const int valid = min(kBN, n_tokens - j * kBN);
            uint32_t s[kBN];
            tmem_ld128_sync(s_addr, s);
            if (valid < kBN) {
#pragma unroll
                for (int c = 0; c < kBN; ++c)
                    if (c >= valid) s[c] = __float_as_uint(-INFINITY);
            }
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < kBN; c += 2)
                mx[(c >> 1) & 3] = fmax3(mx[(c >> 1) & 3], __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
            const float m_tile = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale_log2;
            if (j == 0) {
                m_ref = m_tile;
            } else {
                // Lazy rescale, warp by warp (a warp reaches only its own 32 TMEM lanes).  O_t
                // holds exactly PV_t(0 .. j-1) here: S_t(j) was issued after PV_t(j-1), and
                // PV_t(j) waits for this warpgroup's arrival below.
                const bool grow = m_tile > m_ref + kRescaleSlack;
                if (__any_sync(0xffffffffu, grow)) {
                    const float alpha = grow ? exp2_approx(m_ref - m_tile) : 1.0f;
                    for (int c = 0; c < head_dim; c += 16) {
                        uint32_t o[16];
                        tmem_ld16_sync(o_addr + c, o);
#pragma unroll
                        for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st16(o_addr + c, o);
                    }
                    if (grow) {
                        l *= alpha;
                        m_ref = m_tile;
                    }
                }
            }
            // P_t(j) over S_t(j)'s columns 64..127, all of whose S values are in registers:
            // keys 64..127 to columns 96..127, then keys 0..63 to columns 64..95.
            const uint64_t scale2 = f32x2_pack(scale_log2, scale_log2), neg_m2 = f32x2_pack(-m_ref, -m_ref);
            l += half_weights(*reinterpret_cast<const uint32_t(*)[64]>(s + 64), scale2, neg_m2, s_addr + kPCol + 32u);
            l += half_weights(*reinterpret_cast<const uint32_t(*)[64]>(s), scale2, neg_m2, s_addr + kPCol);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(p_full0 + 8u * t);
        }
        // Epilogue: O_t / l once the last product has landed.
        if (ok && mbar_wait(o_done, 0, abort_flag, status, wait_ns)) {
            tc_fence_after();
            const int row = m0 + kBM * t + r;
            const float inv = 1.0f / l;
            for (int c = 0; c < head_dim; c += 16) {
                uint32_t o[16];
                tmem_ld16_sync(o_addr + c, o);
                if (row < n_tokens) {
                    const int64_t off = (static_cast<int64_t>(h) * n_tokens + row) * head_dim + c;
                    if (OUT_BF16) {
                        uint32_t w[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const __nv_bfloat162 v2 = __floats2bfloat162_rn(__uint_as_float(o[2 * e]) * inv,
                                                                            __uint_as_float(o[2 * e + 1]) * inv);
                            w[e] = *reinterpret_cast<const uint32_t*>(&v2);
                        }
                        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out) + off);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    } else {
                        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + off);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                                 __uint_as_float(o[4 * e + 2]) * inv,
                                                 __uint_as_float(o[4 * e + 3]) * inv);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int NBOX, bool BF16>
cudaError_t launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, void* out, int heads,
                   int n_tokens, int head_dim, float scale_log2, int* status, uint64_t wait_ns,
                   cudaStream_t stream) {
    using L = AttnLayout<NBOX>;
    cudaError_t e = cudaFuncSetAttribute(anchor_attention_kernel<NBOX, BF16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::smem_bytes);
    if (e != cudaSuccess) return e;
    const int q_blocks = (n_tokens + kQTiles * kBM - 1) / (kQTiles * kBM);
    anchor_attention_kernel<NBOX, BF16><<<heads * q_blocks, kAttnThreads, L::smem_bytes, stream>>>(
        tq, tk, tv, out, n_tokens, head_dim, scale_log2, status, wait_ns);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_anchor_attention(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                    void* out, bool out_bf16, int heads, int64_t n_tokens, int head_dim,
                                    float scale_log2, int* status, uint64_t wait_ns, cudaStream_t stream) {
    const int n = static_cast<int>(n_tokens);
    if (head_dim_atoms(head_dim) == 1)
        return out_bf16 ? launch<1, true>(tm_q, tm_k, tm_v, out, heads, n, head_dim, scale_log2, status, wait_ns, stream)
                        : launch<1, false>(tm_q, tm_k, tm_v, out, heads, n, head_dim, scale_log2, status, wait_ns, stream);
    return out_bf16 ? launch<2, true>(tm_q, tm_k, tm_v, out, heads, n, head_dim, scale_log2, status, wait_ns, stream)
                    : launch<2, false>(tm_q, tm_k, tm_v, out, heads, n, head_dim, scale_log2, status, wait_ns, stream);
}

}  // namespace la
