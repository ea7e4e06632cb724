// Shared declarations of the lin_attn kernels and their host-side launchers.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace la {

// Token tile of the KV reduction (rows per pipeline stage of the tensor-core kernel, and
// the unit of the work split).
constexpr int kKvTile = 64;
// Token tile of the tensor-core apply kernel (MMA M).
constexpr int kApplyTile = 128;
// Work chunks of the KV reduction.  Each head's 64-token tiles are cut into k contiguous
// chunks of equal size (+-1 tile), at the same token boundaries for every head:
// k = min(floor(152 / H), tiles per head, 150), at least 1, and G = k H chunks in head
// order (chunk c is part c % k of head c / k).  Each chunk is summed by one CTA and leaves
// one partial KV.  With every head cut at the same tokens, the CTAs that run at the same
// time walk the same token rows of all heads, which keeps reads of token-major [N, H, D]
// activations on whole DRAM rows.  k and G are constants of the shape (152 = one chunk per
// SM of a 152-SM part), never read from the device, so the summation order is fixed by the
// shape.
constexpr int kChunks = 152;
constexpr int kChunksPerHeadCap = 150;  // k <= 150 keeps a head under kMaxSegments partials
constexpr int kMaxSegments = 160;       // partials per head the reduction can add

struct KvPlan {
    int64_t tiles_per_head;  // ceil(N / kKvTile)
    int64_t total_tiles;     // H * tiles_per_head
    int chunks;              // G = k H
    int per_head;            // k: chunks (and partials) per head
    int seg_stride;          // partial slots per head (= k)
};

__host__ __device__ inline int kv_chunks_per_head(int heads, int64_t tiles_per_head) {
    int64_t k = kChunks / heads;
    if (k > tiles_per_head) k = tiles_per_head;
    if (k > kChunksPerHeadCap) k = kChunksPerHeadCap;
    return k < 1 ? 1 : static_cast<int>(k);
}
__host__ __device__ inline KvPlan kv_plan(int heads, int64_t n_tokens) {
    KvPlan p;
    p.tiles_per_head = (n_tokens + kKvTile - 1) / kKvTile;
    p.total_tiles = p.tiles_per_head * heads;
    p.per_head = kv_chunks_per_head(heads, p.tiles_per_head);
    p.chunks = p.per_head * heads;
    p.seg_stride = p.per_head;
    return p;
}
// First tile of chunk c (chunk c covers [chunk_begin(c), chunk_begin(c + 1))).
__host__ __device__ inline int64_t chunk_begin(const KvPlan& p, int64_t c) {
    const int64_t h = c / p.per_head, g = c % p.per_head;
    return h * p.tiles_per_head + g * p.tiles_per_head / p.per_head;
}
// The chunk that holds tile t.
__host__ __device__ inline int64_t chunk_of_tile(const KvPlan& p, int64_t t) {
    const int64_t h = t / p.tiles_per_head, lt = t % p.tiles_per_head;
    return h * p.per_head + ((lt + 1) * p.per_head - 1) / p.tiles_per_head;
}
// Partial slot of (head h, chunk c) and the number of partials of head h.
__host__ __device__ inline int segment_of(const KvPlan& p, int h, int64_t c) {
    return static_cast<int>(c - static_cast<int64_t>(h) * p.per_head);
}
__host__ __device__ inline int segments_of_head(const KvPlan& p, int) { return p.per_head; }
// Largest seg_stride any n_tokens can produce for `heads` (scratch sizing).
__host__ __device__ inline int kv_seg_stride_bound(int heads) {
    return kv_chunks_per_head(heads, static_cast<int64_t>(kChunksPerHeadCap));
}

// Work of one launch of the KV reduction: heads [h0, h0 + hc) of the layer (the K/V
// pointers and tensor maps start at head h0), i.e. tiles [t_lo, t_hi) of chunks
// [c_lo, c_hi].
struct KvLaunch {
    int h0;
    int64_t t_lo, t_hi;
    int64_t c_lo;
    int n_chunks;
};
__host__ __device__ inline KvLaunch kv_launch(const KvPlan& p, int h0, int hc) {
    KvLaunch l;
    l.h0 = h0;
    l.t_lo = h0 * p.tiles_per_head;
    l.t_hi = (h0 + hc) * p.tiles_per_head;
    l.c_lo = chunk_of_tile(p, l.t_lo);
    l.n_chunks = static_cast<int>(chunk_of_tile(p, l.t_hi - 1) - l.c_lo + 1);
    return l;
}

// Element strides of a [.., N, .., D] activation (Q, K, V or out): row n of head h starts
// at h * head + n * token.  Head-major [1, H, N, D]: (N*D, D).  Token-major [1, N, H, D],
// the projection layout of the model: (D, H*D).
struct Strides {
    int64_t head;
    int64_t token;
};

// Number of 64-wide column blocks ("atoms") that cover the head dim: 1 for D <= 64, else 2.
__host__ __device__ constexpr int head_dim_atoms(int head_dim) { return (head_dim + 63) / 64; }

// Bytes of one head's three-term BF16 image of KV^T in the 128-byte-swizzled K-major
// layout the apply kernel's MMA reads straight from shared memory.
__host__ __device__ constexpr int64_t kv_image_bytes(int head_dim) {
    return 3ll * head_dim_atoms(head_dim) * head_dim * 128;
}

// Sets the calling thread's last-error text (lin_attn_last_error); returns `code`.
int record_error(int code, const char* msg);

// Launch `kernel` with programmatic stream serialisation: it may start while the previous
// kernel of the stream finishes.  Every kernel launched this way calls grid_dependency_wait
// before it touches memory an earlier kernel of the stream may still be using.
template <typename... Params, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// The producer step fused into the tensor-core kernels (ReLU + interleaved RoPE on the
// loaded Q / K tiles, the normaliser from the activated un-rotated copies).
//   cos, sin : FP32 [N][D/2] rotation tables (pair p of token n is turned by cos/sin[n][p])
//   ksum_partial : FP64 [H][seg_stride][kKsumGroups][D] per-chunk, per-row-group column
//                  sums of relu(K) (scratch)
//   ksum : FP32 [H][D] reduced column sums (scratch; read by the apply)
// Row groups of the fused KV kernel's transform (one column-sum partial each).
constexpr int kKsumGroups = 16;
struct ProducerArgs {
    const float* cos;
    const float* sin;
    double* ksum_partial;
    float* ksum;
    int n_tokens;
};
// Added to every normaliser denominator (den = relu(q) . sum relu(k) + kDenEps).
constexpr float kDenEps = 1e-6f;

// Producer step on one 16-byte chunk (8 BF16 values = 4 rotation pairs) of a Q or K row:
// ReLU, then each pair (x0, x1) is turned by (c, s) as (x0 c - x1 s, x0 s + x1 c) with
// binary32 products and sums in exactly this order, rounded once to BF16 (nearest-even).
// The rotation stays on scalar round-to-nearest intrinsics, which the compiler never fuses
// into a multiply-add (a paired multiply feeding a paired add can be fused, which moves
// exact ties).  The activated (un-rotated) values come back for the normaliser as paired
// registers act0[h] = {x0 of pairs 2h, 2h + 1} (chunk columns 4h, 4h + 2) and
// act1[h] = {x1 of the same pairs} (columns 4h + 1, 4h + 3).
__device__ __forceinline__ void rope_chunk(uint4& w, const float4 c4, const float4 s4, uint64_t (&act0)[2],
                                           uint64_t (&act1)[2]) {
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t outw[4];
    float x0[4], x1[4];
    const float cs[4] = {c4.x, c4.y, c4.z, c4.w};
    const float sn[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        x0[j] = fmaxf(__uint_as_float(in[j] << 16), 0.f);
        x1[j] = fmaxf(__uint_as_float(in[j] & 0xFFFF0000u), 0.f);
        const float y0 = __fsub_rn(__fmul_rn(x0[j], cs[j]), __fmul_rn(x1[j], sn[j]));
        const float y1 = __fadd_rn(__fmul_rn(x0[j], sn[j]), __fmul_rn(x1[j], cs[j]));
        const __nv_bfloat162 y = __floats2bfloat162_rn(y0, y1);
        outw[j] = *reinterpret_cast<const uint32_t*>(&y);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        act0[h] = f32x2_pack(x0[2 * h], x0[2 * h + 1]);
        act1[h] = f32x2_pack(x1[2 * h], x1[2 * h + 1]);
    }
    w = make_uint4(outw[0], outw[1], outw[2], outw[3]);
}

// ---------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error.  `partial` is the base of the layer's
// [H][seg_stride][D][D] partial buffer (head 0); the K/V maps/pointers start at head h0.

// KV partial sums on tensor cores (BF16 x BF16 -> FP32).  The tensor maps index
// (column, token, head) or, if token_major, (column, head, token).  `lossless` promotes
// the tensor-core sums into FP32 registers every tile instead of every 4 tiles.
// With `producer` (fused path) tm_tables holds the maps of the two rotation tables (2-D,
// (D/2, N), box (D/2, 64), no swizzle).
cudaError_t launch_kv_partial_tc(const CUtensorMap& tm_k, const CUtensorMap& tm_v, float* partial, int64_t n_tokens,
                                 int head_dim, const KvPlan& plan, const KvLaunch& work, bool token_major,
                                 bool lossless, int* status, uint64_t wait_ns, cudaStream_t stream,
                                 const ProducerArgs* producer = nullptr, const CUtensorMap* tm_tables = nullptr);

// Fixed-order pairwise reduction of each head's partials for heads [h0, h0 + hc):
// kv[h][i][j] (FP32) and, if kv_image != nullptr, its three-term BF16 image for the
// tensor-core apply.  kv / kv_image are the layer's base pointers (head 0).
cudaError_t launch_kv_finalize(const float* partial, float* kv, uint8_t* kv_image, int h0, int hc, int head_dim,
                               const KvPlan& plan, cudaStream_t stream, const ProducerArgs* producer = nullptr);

// out = (Q . KV) * (1 / den) on tensor cores, KV as three BF16 terms (maps as above).
cudaError_t launch_apply_tc(const CUtensorMap& tm_q, const CUtensorMap& tm_out, const uint8_t* kv_image,
                            const float* den, int heads, int64_t n_tokens, int head_dim, bool out_bf16,
                            bool token_major, int grid, int* status, uint64_t wait_ns, cudaStream_t stream);

// Softmax anchor attention (flash forward): out = softmax(scale * Q K^T) V per head, no
// mask.  Maps over [H][N][D] BF16: Q box (64, 128), K and V boxes (64, 64); scale_log2 =
// scale * log2(e).
// Second GEMM of the fused producer path, computed as out^T = KV^T Q_rot^T with the KV
// image in TMEM.  tm_q as for launch_apply_tc; tm_out_t maps out with a (32 features,
// 32 tokens) box and no swizzle; both index (column, head, token) if token_major.
cudaError_t launch_apply_fused_tc(const CUtensorMap& tm_q, const CUtensorMap& tm_out_t, const uint8_t* kv_image,
                                  int heads, int64_t n_tokens, int head_dim, bool out_bf16, bool token_major, int grid,
                                  int* status, uint64_t wait_ns, cudaStream_t stream, const ProducerArgs& producer);

cudaError_t launch_anchor_attention(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                    void* out, bool out_bf16, int heads, int64_t n_tokens, int head_dim,
                                    float scale_log2, int* status, uint64_t wait_ns, cudaStream_t stream);

}  // namespace la
