// First GEMM of SANA-Video linear attention: KV[h] = K_rot[h]^T . V[h], reduced over tokens.
//
// Page "PR #35728 完整报告 - [diffusion] Accelerate SANA-Video linear attention in
// quality=high", 关键源码片段: the site runs the first GEMM as a BF16 bmm with FP32
// accumulation/output ('high'); the model's fallback chain upcasts both operands to FP32
// first ('lossless').  The token axis is cut into S splits per head (S fixed by the shape);
// each split's D x D partial sum goes to scratch, and kv_finalize adds the S partials in a
// fixed pairwise order, so the result is the same on every run.
#include <cuda_bf16.h>

#include "lin_attn_internal.cuh"
#include "ptx.cuh"

namespace la {
namespace {

// ============================================================================ tensor cores
// Warp roles: warp 0 issues TMA loads, warp 1 issues tcgen05.mma, warps 2..5 drain the
// TMEM accumulator to scratch.  Per stage, one 64-token tile of K and of V is loaded with
// 128-byte swizzle as [token][64 head-dim columns] boxes - exactly the MN-major canonical
// layout of the MMA operands A = K^T (M = head-dim row i) and B = V (N = head-dim column j),
// with K = tokens.  M is always 128 (head dims up to 128; rows i >= D are zero).
constexpr int kKvStages = 6;
constexpr int kKvThreads = 192;
constexpr int kKvPromoteTiles = 4;  // tiles per tensor-core sub-chunk (256 tokens)
constexpr uint32_t kKvAtomBytes = kKvTile * 128;  // one box: 64 token rows x 128 bytes

template <int NBOX>
struct KvLayout {
    static constexpr uint32_t a_bytes = 2 * kKvAtomBytes;  // A = K^T: 2 atoms cover M = 128
    static constexpr uint32_t b_bytes = NBOX * kKvAtomBytes;
    static constexpr uint32_t stage_bytes = a_bytes + b_bytes;
    static constexpr uint32_t bar_offset = kKvStages * stage_bytes;
    static constexpr uint32_t smem_bytes = bar_offset + 256 + 1024;  // + barriers + alignment slack
};

template <int NBOX>
__global__ void __launch_bounds__(kKvThreads, 1)
    kv_partial_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         float* __restrict__ partial, int heads, int n_tokens, int head_dim, int chunk,
                         int splits, int* status) {
    using L = KvLayout<NBOX>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);

    const uint32_t bars = base + L::bar_offset;
    const uint32_t full0 = bars;                          // [kKvStages]
    const uint32_t empty0 = bars + 8u * kKvStages;        // [kKvStages]
    const uint32_t acc_full0 = bars + 16u * kKvStages;    // [2]
    const uint32_t acc_empty0 = acc_full0 + 16u;          // [2]
    const uint32_t drain_bar = acc_empty0 + 16u;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base_ptr + L::bar_offset + 192);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + L::bar_offset + 200);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int units = heads * splits;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kKvStages; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, 1);
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
        for (uint32_t idx = threadIdx.x; idx < kKvStages * (kKvAtomBytes / 16); idx += blockDim.x) {
            const uint32_t st = idx / (kKvAtomBytes / 16), off = idx % (kKvAtomBytes / 16);
            *reinterpret_cast<uint4*>(base_ptr + st * L::stage_bytes + kKvAtomBytes + off * 16) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), 256);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- producer
            uint32_t it = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
                const int h = u / splits, s = u % splits;
                const int t0 = s * chunk;
                const int t1 = min(t0 + chunk, n_tokens);
                const int ntiles = (t1 - t0 + kKvTile - 1) / kKvTile;
                for (int k = 0; k < ntiles; ++k, ++it) {
                    const uint32_t st = it % kKvStages, ph = (it / kKvStages) & 1u;
                    if (!mbar_wait(empty0 + 8u * st, ph ^ 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t a = base + st * L::stage_bytes;
                    const uint32_t b = a + L::a_bytes;
                    mbar_arrive_expect_tx(full0 + 8u * st, 2u * NBOX * kKvAtomBytes);
#pragma unroll
                    for (int x = 0; x < NBOX; ++x) {
                        tma_load_3d(a + x * kKvAtomBytes, &tm_k, full0 + 8u * st, 64 * x, t0 + k * kKvTile, h);
                        tma_load_3d(b + x * kKvAtomBytes, &tm_v, full0 + 8u * st, 64 * x, t0 + k * kKvTile, h);
                    }
                }
            }
            if (!ok) {
                // Let the loads already issued land before shared memory goes away.
                const uint32_t first = it > kKvStages ? it - kKvStages : 0;
                for (uint32_t j = first; j < it; ++j)
                    mbar_wait_drain(full0 + 8u * (j % kKvStages), (j / kKvStages) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            // Each split is accumulated in sub-chunks of kKvPromoteTiles tiles, alternating
            // between two TMEM accumulators; the epilogue adds every finished sub-chunk into
            // FP32 registers (round-to-nearest), so tensor-core accumulation never runs over
            // more than kKvPromoteTiles * 64 tokens.
            constexpr uint32_t idesc = make_idesc_bf16_f32(128, 64 * NBOX, true, true);
            uint32_t it = 0, sub = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
                const int s = u % splits;
                const int t0 = s * chunk;
                const int t1 = min(t0 + chunk, n_tokens);
                const int ntiles = (t1 - t0 + kKvTile - 1) / kKvTile;
                for (int k0 = 0; ok && k0 < ntiles; k0 += kKvPromoteTiles, ++sub) {
                    const int k1 = min(k0 + kKvPromoteTiles, ntiles);
                    const uint32_t buf = sub & 1u;
                    if (!mbar_wait(acc_empty0 + 8u * buf, ((sub >> 1) & 1u) ^ 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + buf * 128u;
                    for (int k = k0; k < k1; ++k, ++it) {
                        const uint32_t st = it % kKvStages, ph = (it / kKvStages) & 1u;
                        if (!mbar_wait(full0 + 8u * st, ph, abort_flag, status)) {
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
            }
            mma_commit(drain_bar);
            mbar_wait_drain(drain_bar, 0);
        }
    } else {
        // ---------------- epilogue: TMEM lanes 32q..32q+31 = rows i of the partial KV.
        // Thread i keeps its row of the split's running sum in registers.
        const int q = warp & 3;
        const int i = 32 * q + lane;
        uint32_t sub = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
            const int h = u / splits, s = u % splits;
            const int t0 = s * chunk;
            const int t1 = min(t0 + chunk, n_tokens);
            const int ntiles = (t1 - t0 + kKvTile - 1) / kKvTile;
            float acc[64 * NBOX];
#pragma unroll
            for (int c = 0; c < 64 * NBOX; ++c) acc[c] = 0.f;
            for (int k0 = 0; k0 < ntiles; k0 += kKvPromoteTiles, ++sub) {
                const uint32_t buf = sub & 1u;
                if (!mbar_wait(acc_full0 + 8u * buf, (sub >> 1) & 1u, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * 128u;
#pragma unroll
                for (int c = 0; c < 4 * NBOX; ++c) {
                    if (16 * c < head_dim) {
                        uint32_t r[16];
                        tmem_ld16_sync(taddr + 16u * c, r);
#pragma unroll
                        for (int e = 0; e < 16; ++e) acc[16 * c + e] += __uint_as_float(r[e]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty0 + 8u * buf);
            }
            if (!ok) break;
            if (i < head_dim) {
                float* dst = partial + ((static_cast<int64_t>(h) * splits + s) * head_dim + i) * head_dim;
#pragma unroll
                for (int c = 0; c < 4 * NBOX; ++c) {
                    if (16 * c < head_dim) {
                        float4* o = reinterpret_cast<float4*>(dst + 16 * c);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            o[e] = make_float4(acc[16 * c + 4 * e], acc[16 * c + 4 * e + 1], acc[16 * c + 4 * e + 2],
                                               acc[16 * c + 4 * e + 3]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// ============================================================================ CUDA cores
// 'lossless': both operands upcast from BF16 to FP32 (exact), FP32 FMA, one block per
// (split, head); thread (ti, tj) owns KV rows ti + 16a and columns tj + 16b.
constexpr int kFfmaKvRows = 32;

template <int C>
__global__ void __launch_bounds__(256) kv_partial_ffma_kernel(const uint16_t* __restrict__ k,
                                                              const uint16_t* __restrict__ v,
                                                              float* __restrict__ partial, int n_tokens,
                                                              int chunk, int splits) {
    constexpr int D = 16 * C;
    __shared__ float ks[kFfmaKvRows][D];
    __shared__ float vs[kFfmaKvRows][D];
    const int s = blockIdx.x, h = blockIdx.y;
    const int t0 = s * chunk;
    const int t1 = min(t0 + chunk, n_tokens);
    const int ti = threadIdx.x & 15, tj = threadIdx.x >> 4;
    const uint16_t* kh = k + static_cast<int64_t>(h) * n_tokens * D;
    const uint16_t* vh = v + static_cast<int64_t>(h) * n_tokens * D;

    float acc[C][C];
#pragma unroll
    for (int a = 0; a < C; ++a)
#pragma unroll
        for (int b = 0; b < C; ++b) acc[a][b] = 0.f;

    for (int n0 = t0; n0 < t1; n0 += kFfmaKvRows) {
        const int rows = min(kFfmaKvRows, t1 - n0);
        __syncthreads();
        for (int idx = threadIdx.x; idx < kFfmaKvRows * (D / 8); idx += 256) {
            const int r = idx / (D / 8), c = idx % (D / 8);
            uint4 kw = make_uint4(0, 0, 0, 0), vw = make_uint4(0, 0, 0, 0);
            if (r < rows) {
                kw = *reinterpret_cast<const uint4*>(kh + static_cast<int64_t>(n0 + r) * D + 8 * c);
                vw = *reinterpret_cast<const uint4*>(vh + static_cast<int64_t>(n0 + r) * D + 8 * c);
            }
            const uint32_t kk[4] = {kw.x, kw.y, kw.z, kw.w};
            const uint32_t vv[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                ks[r][8 * c + 2 * e] = __uint_as_float(kk[e] << 16);
                ks[r][8 * c + 2 * e + 1] = __uint_as_float(kk[e] & 0xFFFF0000u);
                vs[r][8 * c + 2 * e] = __uint_as_float(vv[e] << 16);
                vs[r][8 * c + 2 * e + 1] = __uint_as_float(vv[e] & 0xFFFF0000u);
            }
        }
        __syncthreads();
        for (int r = 0; r < rows; ++r) {
            float kr[C], vr[C];
#pragma unroll
            for (int a = 0; a < C; ++a) kr[a] = ks[r][ti + 16 * a];
#pragma unroll
            for (int b = 0; b < C; ++b) vr[b] = vs[r][tj + 16 * b];
#pragma unroll
            for (int a = 0; a < C; ++a)
#pragma unroll
                for (int b = 0; b < C; ++b) acc[a][b] = fmaf(kr[a], vr[b], acc[a][b]);
        }
    }
    float* dst = partial + (static_cast<int64_t>(h) * splits + s) * D * D;
#pragma unroll
    for (int a = 0; a < C; ++a)
#pragma unroll
        for (int b = 0; b < C; ++b) dst[(ti + 16 * a) * D + tj + 16 * b] = acc[a][b];
}

// ============================================================================ reduction
// kv[h][e] = pairwise tree over the S partials: level w adds partial s + w into s for every
// s that is a multiple of 2w.  The shape fixes S and so the order.  Also writes the
// three-term BF16 image of KV^T for the tensor-core apply: row j, column i of term t sits
// in 64-column atom i / 64, in the 128-byte-swizzled K-major layout (16-byte chunk
// (i % 64) / 8 of row j stored at chunk position ((i % 64) / 8) ^ (j % 8)).
__global__ void __launch_bounds__(256) kv_finalize_kernel(const float* __restrict__ partial,
                                                          float* __restrict__ kv, uint8_t* __restrict__ image,
                                                          int head_dim, int splits) {
    const int h = blockIdx.y;
    const int dd = head_dim * head_dim;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= dd) return;
    const float* p = partial + static_cast<int64_t>(h) * splits * dd + e;
    float vals[kMaxSplits];
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) vals[s] = s < splits ? p[static_cast<int64_t>(s) * dd] : 0.f;
#pragma unroll
    for (int w = 1; w < kMaxSplits; w *= 2) {
#pragma unroll
        for (int s = 0; s + w < kMaxSplits; s += 2 * w)
            if (s + w < splits) vals[s] = vals[s] + vals[s + w];
    }
    const float x = vals[0];
    kv[static_cast<int64_t>(h) * dd + e] = x;
    if (image == nullptr) return;

    const __nv_bfloat16 hi = __float2bfloat16_rn(x);
    const float r1 = x - __bfloat162float(hi);  // exact
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);  // exact
    const __nv_bfloat16 lo = __float2bfloat16_rn(r2);

    const int i = e / head_dim, j = e % head_dim;
    const int atoms = head_dim_atoms(head_dim);
    const int64_t term_bytes = static_cast<int64_t>(atoms) * head_dim * 128;
    const int a = i >> 6, c = i & 63;
    const int64_t off = static_cast<int64_t>(a) * head_dim * 128 + j * 128 + ((((c >> 3) ^ (j & 7))) << 4) + (c & 7) * 2;
    uint8_t* img = image + static_cast<int64_t>(h) * 3 * term_bytes + off;
    *reinterpret_cast<__nv_bfloat16*>(img) = hi;
    *reinterpret_cast<__nv_bfloat16*>(img + term_bytes) = mid;
    *reinterpret_cast<__nv_bfloat16*>(img + 2 * term_bytes) = lo;
}

template <int NBOX>
cudaError_t launch_tc(const CUtensorMap& tm_k, const CUtensorMap& tm_v, float* partial, int heads, int n_tokens,
                      int head_dim, SplitPlan plan, int grid, int* status, cudaStream_t stream) {
    using L = KvLayout<NBOX>;
    cudaError_t e = cudaFuncSetAttribute(kv_partial_tc_kernel<NBOX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::smem_bytes);
    if (e != cudaSuccess) return e;
    kv_partial_tc_kernel<NBOX><<<grid, kKvThreads, L::smem_bytes, stream>>>(
        tm_k, tm_v, partial, heads, n_tokens, head_dim, static_cast<int>(plan.chunk), plan.splits, status);
    return cudaGetLastError();
}

template <int C>
cudaError_t launch_ffma(const uint16_t* k, const uint16_t* v, float* partial, int heads, int n_tokens,
                        SplitPlan plan, cudaStream_t stream) {
    dim3 grid(plan.splits, heads);
    kv_partial_ffma_kernel<C><<<grid, 256, 0, stream>>>(k, v, partial, n_tokens, static_cast<int>(plan.chunk),
                                                       plan.splits);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kv_partial_tc(const CUtensorMap& tm_k, const CUtensorMap& tm_v, float* partial, int heads,
                                 int64_t n_tokens, int head_dim, SplitPlan plan, int grid, int* status,
                                 cudaStream_t stream) {
    const int units = heads * plan.splits;
    if (grid > units) grid = units;
    if (head_dim_atoms(head_dim) == 1)
        return launch_tc<1>(tm_k, tm_v, partial, heads, static_cast<int>(n_tokens), head_dim, plan, grid, status,
                            stream);
    return launch_tc<2>(tm_k, tm_v, partial, heads, static_cast<int>(n_tokens), head_dim, plan, grid, status,
                        stream);
}

cudaError_t launch_kv_partial_ffma(const uint16_t* k, const uint16_t* v, float* partial, int heads,
                                   int64_t n_tokens, int head_dim, SplitPlan plan, cudaStream_t stream) {
    const int n = static_cast<int>(n_tokens);
    switch (head_dim / 16) {
        case 1: return launch_ffma<1>(k, v, partial, heads, n, plan, stream);
        case 2: return launch_ffma<2>(k, v, partial, heads, n, plan, stream);
        case 3: return launch_ffma<3>(k, v, partial, heads, n, plan, stream);
        case 4: return launch_ffma<4>(k, v, partial, heads, n, plan, stream);
        case 5: return launch_ffma<5>(k, v, partial, heads, n, plan, stream);
        case 6: return launch_ffma<6>(k, v, partial, heads, n, plan, stream);
        case 7: return launch_ffma<7>(k, v, partial, heads, n, plan, stream);
        case 8: return launch_ffma<8>(k, v, partial, heads, n, plan, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_kv_finalize(const float* partial, float* kv, uint8_t* kv_image, int heads, int head_dim,
                               int splits, cudaStream_t stream) {
    const int dd = head_dim * head_dim;
    dim3 grid((dd + 255) / 256, heads);
    kv_finalize_kernel<<<grid, 256, 0, stream>>>(partial, kv, kv_image, head_dim, splits);
    return cudaGetLastError();
}

}  // namespace la
