// SANA-Video 2.0 softmax anchor attention on tensor cores (flash-attention forward).
//
// Page "[sglang] SANA-Video 2.0 anchor attention의 FP32 upcast 제거로 720p 생성 52%
// 단축하기" (PR #49219), section 코드 분석, 2. GatedSoftmaxAttention: the anchor layer is
// F.scaled_dot_product_attention(q, k, v, dropout_p=0.0) on BF16 [B, H, N, D] tensors (no
// mask, default scale 1/sqrt(D)); the page's 'high' tier hands BF16 Q/K/V to a flash
// kernel.  Here, per head and per 128-query tile:
//     S = Q K^T (tcgen05, FP32 in TMEM), P = exp2(S * scale * log2 e - m) (BF16 in shared
//     memory), O += P V (tcgen05, FP32 in TMEM), out = O / sum(P)
// with the running maximum m kept per row and O rescaled only when a row's maximum grows
// by more than 8 (in log2 units) - the weights stay below 2^8, and O / sum(P) is exact for
// any reference m - so the rescale (a TMEM read-modify-write) is rare.
#include <cuda_bf16.h>

#include "lin_attn_internal.cuh"
#include "ptx.cuh"

namespace la {
namespace {

constexpr int kBM = 128;                  // query rows per CTA tile (MMA M, one row per thread)
constexpr int kBN = 64;                   // keys per iteration
constexpr int kAttnStages = 4;            // K/V ring
constexpr int kAttnThreads = 192;         // warp 0 TMA, warp 1 MMA, warps 2..5 softmax/epilogue
constexpr uint32_t kQAtom = kBM * 128;    // 16 KB: 128 rows x 64 columns BF16 (128-byte swizzle)
constexpr uint32_t kKVAtom = kBN * 128;   // 8 KB: 64 rows x 64 columns BF16
constexpr uint32_t kPBytes = kBM * 128;   // 16 KB: P tile, 128 queries x 64 keys BF16
constexpr float kRescaleSlack = 8.0f;     // rescale O when a row maximum grows by more than this

template <int NBOX>
struct AttnLayout {
    static constexpr uint32_t q_bytes = NBOX * kQAtom;
    static constexpr uint32_t stage_bytes = 2 * NBOX * kKVAtom;  // K tile + V tile
    static constexpr uint32_t kv_offset = q_bytes;
    static constexpr uint32_t p_offset = kv_offset + kAttnStages * stage_bytes;
    static constexpr uint32_t bar_offset = p_offset + 2 * kPBytes;
    static constexpr uint32_t smem_bytes = bar_offset + 256 + 1024;
};

// TMEM columns: S buffers at 0 and 64, O at 128 (up to 128 columns).
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kOCol = 128;

template <int NBOX, bool OUT_BF16>
__global__ void __launch_bounds__(kAttnThreads, 1)
    anchor_attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, void* __restrict__ out, int n_tokens,
                            int head_dim, float scale_log2, int* status) {
    using L = AttnLayout<NBOX>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);

    const uint32_t bars = base + L::bar_offset;
    const uint32_t q_full = bars;
    const uint32_t kv_full0 = bars + 8u;                         // [stages]
    const uint32_t kv_empty0 = kv_full0 + 8u * kAttnStages;      // [stages]
    const uint32_t s_full0 = kv_empty0 + 8u * kAttnStages;       // [2] S(j) in TMEM buffer j % 2
    const uint32_t p_full0 = s_full0 + 16u;                      // [2] P(j) written (and S(j) read)
    const uint32_t p_empty0 = p_full0 + 16u;                     // [2] PV(j) done reading P(j)
    const uint32_t o_ready = p_empty0 + 16u;                     // one phase per PV
    const uint32_t o_done = o_ready + 8u;                         // the last PV has landed
    const uint32_t drain_bar = o_done + 8u;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + L::bar_offset + 192);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + L::bar_offset + 200);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int q_tiles = (n_tokens + kBM - 1) / kBM;
    const int h = blockIdx.x / q_tiles;
    const int m0 = (blockIdx.x % q_tiles) * kBM;
    const int n_kv = (n_tokens + kBN - 1) / kBN;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < kAttnStages; ++s) {
            mbar_init(kv_full0 + 8u * s, 1);
            mbar_init(kv_empty0 + 8u * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(s_full0 + 8u * b, 1);
            mbar_init(p_full0 + 8u * b, 128);
            mbar_init(p_empty0 + 8u * b, 1);
        }
        mbar_init(o_ready, 1);
        mbar_init(o_done, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- producer: the Q tile once, then K/V tiles through the ring
            const uint64_t pol_q = policy_evict_first();
            mbar_arrive_expect_tx(q_full, NBOX * kQAtom);
#pragma unroll
            for (int x = 0; x < NBOX; ++x) tma_load_3d_hint(base + x * kQAtom, &tm_q, q_full, 64 * x, m0, h, pol_q);
            bool ok = true;
            uint32_t j = 0;
            for (; j < static_cast<uint32_t>(n_kv); ++j) {
                const uint32_t st = j % kAttnStages, ph = (j / kAttnStages) & 1u;
                if (!mbar_wait(kv_empty0 + 8u * st, ph ^ 1u, abort_flag, status)) {
                    ok = false;
                    break;
                }
                const uint32_t kt = base + L::kv_offset + st * L::stage_bytes;
                const uint32_t vt = kt + NBOX * kKVAtom;
                mbar_arrive_expect_tx(kv_full0 + 8u * st, L::stage_bytes);
#pragma unroll
                for (int x = 0; x < NBOX; ++x) {
                    tma_load_3d(kt + x * kKVAtom, &tm_k, kv_full0 + 8u * st, 64 * x, j * kBN, h);
                    tma_load_3d(vt + x * kKVAtom, &tm_v, kv_full0 + 8u * st, 64 * x, j * kBN, h);
                }
            }
            if (!ok) {
                const uint32_t first = j > kAttnStages ? j - kAttnStages : 0;
                for (uint32_t i = first; i < j; ++i)
                    mbar_wait_drain(kv_full0 + 8u * (i % kAttnStages), (i / kAttnStages) & 1u);
                mbar_wait_drain(q_full, 0);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer: S(0), S(1), then per tile j: PV(j), S(j + 2)
            const uint32_t idesc_s = make_idesc_bf16_f32(kBM, kBN, false, false);      // Q, K both K-major
            const uint32_t idesc_o = make_idesc_bf16_f32(kBM, head_dim, false, true);  // P K-major, V MN-major
            const uint32_t qa = base;
            auto issue_s = [&](uint32_t jj) -> bool {
                const uint32_t st = jj % kAttnStages, ph = (jj / kAttnStages) & 1u;
                if (!mbar_wait(kv_full0 + 8u * st, ph, abort_flag, status)) return false;
                tc_fence_after();
                const uint32_t kt = base + L::kv_offset + st * L::stage_bytes;
                const uint32_t d = tmem + (jj & 1u) * kBN;
#pragma unroll
                for (int ks = 0; ks < 4 * NBOX; ++ks) {
                    const uint32_t x = ks >> 2, off = (ks & 3) * 32u;
                    const uint64_t ad = make_smem_desc(qa + x * kQAtom + off, 16u, 1024u, kSwizzle128B);
                    const uint64_t bd = make_smem_desc(kt + x * kKVAtom + off, 16u, 1024u, kSwizzle128B);
                    mma_bf16(d, ad, bd, idesc_s, ks != 0 ? 1u : 0u);
                }
                mma_commit(s_full0 + 8u * (jj & 1u));
                return true;
            };
            bool ok = mbar_wait(q_full, 0, abort_flag, status);
            if (ok) tc_fence_after();
            for (uint32_t jj = 0; ok && jj < 2 && jj < static_cast<uint32_t>(n_kv); ++jj) ok = issue_s(jj);
            for (uint32_t j = 0; ok && j < static_cast<uint32_t>(n_kv); ++j) {
                const uint32_t b = j & 1u;
                if (!mbar_wait(p_full0 + 8u * b, (j >> 1) & 1u, abort_flag, status)) break;
                tc_fence_after();
                const uint32_t st = j % kAttnStages;
                const uint32_t vt = base + L::kv_offset + st * L::stage_bytes + NBOX * kKVAtom;
                const uint32_t pa = base + L::p_offset + b * kPBytes;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t ad = make_smem_desc(pa + kk * 32u, 16u, 1024u, kSwizzle128B);
                    const uint64_t bd = make_smem_desc(vt + kk * 2048u, kKVAtom, 1024u, kSwizzle128B);
                    mma_bf16(tmem + kOCol, ad, bd, idesc_o, (j | kk) != 0 ? 1u : 0u);
                }
                mma_commit(p_empty0 + 8u * b);
                mma_commit(kv_empty0 + 8u * st);
                mma_commit(o_ready);
                if (j + 1 == static_cast<uint32_t>(n_kv)) mma_commit(o_done);
                if (j + 2 < static_cast<uint32_t>(n_kv)) ok = issue_s(j + 2);
            }
            mma_commit(drain_bar);
            mbar_wait_drain(drain_bar, 0);
        }
    } else {
        // ---------------- softmax and epilogue: thread = query row r of the tile
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; ok && j < n_kv; ++j) {
            const uint32_t b = j & 1u;
            if (!mbar_wait(s_full0 + 8u * b, (j >> 1) & 1u, abort_flag, status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sraw[2][32];
            tmem_ld32_sync(tmem + lane_addr + b * kBN, sraw[0]);
            tmem_ld32_sync(tmem + lane_addr + b * kBN + 32, sraw[1]);
            float t[kBN];
            float tmax = -INFINITY;
            const int valid = min(kBN, n_tokens - j * kBN);  // keys past the end are masked out
#pragma unroll
            for (int c = 0; c < kBN; ++c) {
                t[c] = c < valid ? __uint_as_float(sraw[c >> 5][c & 31]) * scale_log2 : -INFINITY;
                tmax = fmaxf(tmax, t[c]);
            }
            // Lazy rescale: the whole warp rescales together (TMEM access is warp-wide).
            const bool grow = j > 0 && tmax > m_ref + kRescaleSlack;
            if (__any_sync(0xffffffffu, grow)) {
                // O must hold PV(j - 1) before it is rescaled.  S(j) was issued after
                // PV(j - 2) and has landed, so PV(j - 2) is done and the PV count is j - 1 or
                // j: o_ready's parity tells the two apart.
                if (!mbar_wait(o_ready, (j - 1) & 1u, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float alpha = grow ? exp2_approx(m_ref - tmax) : 1.0f;
                for (int c = 0; c < head_dim; c += 16) {
                    uint32_t o[16];
                    tmem_ld16_sync(tmem + lane_addr + kOCol + c, o);
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st16(tmem + lane_addr + kOCol + c, o);
                }
                tmem_st_wait();
                if (grow) {
                    l *= alpha;
                    m_ref = tmax;
                }
            }
            if (j == 0) m_ref = tmax;
            // Weights, their running sum, and the BF16 P row for the next MMA.
            uint32_t pw[kBN / 2];
#pragma unroll
            for (int c = 0; c < kBN; c += 2) {
                const float p0 = exp2_approx(t[c] - m_ref);
                const float p1 = exp2_approx(t[c + 1] - m_ref);
                l += p0;
                l += p1;
                const __nv_bfloat162 pp = __floats2bfloat162_rn(p0, p1);
                pw[c / 2] = *reinterpret_cast<const uint32_t*>(&pp);
            }
            // P buffer b is free once PV(j - 2) has read it.
            if (!mbar_wait(p_empty0 + 8u * b, ((j >> 1) & 1u) ^ 1u, abort_flag, status)) {
                ok = false;
                break;
            }
            const uint32_t prow = base + L::p_offset + b * kPBytes + r * 128u;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint32_t addr = prow + ((static_cast<uint32_t>(c) ^ (r & 7u)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pw[4 * c]),
                             "r"(pw[4 * c + 1]), "r"(pw[4 * c + 2]), "r"(pw[4 * c + 3])
                             : "memory");
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(p_full0 + 8u * b);
        }
        // Epilogue: O / l once the last PV has landed (a barrier of its own: by now the PV
        // count can be one of three values, too many for o_ready's parity).
        if (ok && mbar_wait(o_done, 0, abort_flag, status)) {
            tc_fence_after();
            const int row = m0 + r;
            const float inv = 1.0f / l;
            for (int c = 0; c < head_dim; c += 16) {
                uint32_t o[16];
                tmem_ld16_sync(tmem + lane_addr + kOCol + c, o);
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
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int NBOX, bool BF16>
cudaError_t launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, void* out, int heads,
                   int n_tokens, int head_dim, float scale_log2, int* status, cudaStream_t stream) {
    using L = AttnLayout<NBOX>;
    cudaError_t e = cudaFuncSetAttribute(anchor_attention_kernel<NBOX, BF16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::smem_bytes);
    if (e != cudaSuccess) return e;
    const int q_tiles = (n_tokens + kBM - 1) / kBM;
    anchor_attention_kernel<NBOX, BF16><<<heads * q_tiles, kAttnThreads, L::smem_bytes, stream>>>(
        tq, tk, tv, out, n_tokens, head_dim, scale_log2, status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_anchor_attention(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                    void* out, bool out_bf16, int heads, int64_t n_tokens, int head_dim,
                                    float scale_log2, int* status, cudaStream_t stream) {
    const int n = static_cast<int>(n_tokens);
    if (head_dim_atoms(head_dim) == 1)
        return out_bf16 ? launch<1, true>(tm_q, tm_k, tm_v, out, heads, n, head_dim, scale_log2, status, stream)
                        : launch<1, false>(tm_q, tm_k, tm_v, out, heads, n, head_dim, scale_log2, status, stream);
    return out_bf16 ? launch<2, true>(tm_q, tm_k, tm_v, out, heads, n, head_dim, scale_log2, status, stream)
                    : launch<2, false>(tm_q, tm_k, tm_v, out, heads, n, head_dim, scale_log2, status, stream);
}

}  // namespace la
