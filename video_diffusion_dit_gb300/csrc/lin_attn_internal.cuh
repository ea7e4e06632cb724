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
// ---------------------------------------------------------------- work split
// H heads x T tiles shared out over G CTAs.  k = min(floor(G / H), T, cap) (at least 1)
// CTAs per head take the head's first B tiles (the body), cut into k equal parts (+-1
// tile) at the same tiles for every head, so the CTAs running at the same time walk the
// same token rows of all heads: reads of token-major [N, H, D] activations stay on whole
// DRAM rows, and rotation-table rows fetched for one head are served to the others from
// L2.  The E = G - k H CTAs left over (if any) may share the rest (the tail: tiles [B, T)
// of every head, concatenated head after head) in equal parts.  A tail part that runs
// into another head pays for the switch (a new head's operands, a partial written), so B
// is chosen to minimise the longest part counting `switch_cost` tiles per extra head, and
// the tail is used only where parts are long (T / k >= min_part) and it makes the longest
// part shorter.  Chunk c < k H is part c % k of head c / k's body; chunk k H + e is part e
// of the tail.
//
// Chunks are ranges of a virtual order of the tiles: every head's body (head-major), then
// every head's tail.  A chunk's run of tiles of one head is a segment; a body chunk is one
// segment, a tail chunk one per head it touches.
struct TileSplit {
    int heads;
    int per_head;            // k: body chunks per head
    int tail_chunks;         // E
    int chunks;              // k H + E
    int64_t tiles_per_head;  // T
    int64_t body;            // B (T when there is no tail)
};

// Longest tail part, counting `switch_cost` per head beyond its first, for body length b
// and e parts (e >= 1, b < T).
__host__ __device__ inline int64_t tail_part_cost(int heads, int64_t tiles_per_head, int64_t b, int64_t e,
                                                  int64_t switch_cost) {
    const int64_t tl = tiles_per_head - b, all = heads * tl;
    int64_t most = 0;
    for (int64_t j = 0; j < e; ++j) {
        const int64_t u0 = j * all / e, u1 = (j + 1) * all / e;
        const int64_t cost = (u1 - u0) + switch_cost * ((u1 - 1) / tl - u0 / tl);
        most = cost > most ? cost : most;
    }
    return most;
}

__host__ __device__ inline TileSplit tile_split(int heads, int64_t tiles_per_head, int ctas, int per_head_cap,
                                                int64_t min_part, int64_t switch_cost) {
    TileSplit s;
    s.heads = heads;
    s.tiles_per_head = tiles_per_head;
    int64_t k = ctas / heads;
    if (k > tiles_per_head) k = tiles_per_head;
    if (k > per_head_cap) k = per_head_cap;
    if (k < 1) k = 1;
    s.per_head = static_cast<int>(k);
    s.body = tiles_per_head;
    s.tail_chunks = 0;
    const int64_t spare = static_cast<int64_t>(ctas) - k * heads;
    const int64_t no_tail = (tiles_per_head + k - 1) / k;
    if (spare > 0 && k < tiles_per_head && tiles_per_head / k >= min_part) {
        // Equal costs near B = k (H T + switch_cost * ceil(H / E) * E) / G; the candidates
        // around it are costed exactly and the first cheapest is taken.
        const int64_t extra = switch_cost * ((heads + spare - 1) / spare) * spare;
        const int64_t b0 = k * (heads * tiles_per_head + extra) / ctas;
        int64_t best = -1, best_cost = no_tail;
        for (int64_t b = b0 - 2; b <= b0 + 2; ++b) {
            if (b < k || b >= tiles_per_head) continue;
            const int64_t tail = heads * (tiles_per_head - b), e = spare < tail ? spare : tail;
            const int64_t body_cost = (b + k - 1) / k;
            const int64_t tail_cost = tail_part_cost(heads, tiles_per_head, b, e, switch_cost);
            const int64_t cost = body_cost > tail_cost ? body_cost : tail_cost;
            if (cost < best_cost) {
                best = b;
                best_cost = cost;
            }
        }
        if (best >= 0) {
            const int64_t tail = heads * (tiles_per_head - best);
            s.body = best;
            s.tail_chunks = static_cast<int>(spare < tail ? spare : tail);
        }
    }
    s.chunks = s.per_head * heads + s.tail_chunks;
    return s;
}
// Tiles in the tail of one head (T - B) and in all tails.
__host__ __device__ inline int64_t split_tail_len(const TileSplit& s) { return s.tiles_per_head - s.body; }
// First virtual tile of chunk c, for c in [0, chunks]; chunk c covers [begin(c), begin(c + 1)).
__host__ __device__ inline int64_t split_begin(const TileSplit& s, int64_t c) {
    const int64_t kh = static_cast<int64_t>(s.per_head) * s.heads;
    if (c < kh) return (c / s.per_head) * s.body + (c % s.per_head) * s.body / s.per_head;
    const int64_t all_tails = s.heads * split_tail_len(s);
    return s.heads * s.body + (s.tail_chunks ? (c - kh) * all_tails / s.tail_chunks : 0);
}
// Head and tile (within the head) of virtual tile v.
struct HeadTile {
    int h;
    int64_t tile;
};
__host__ __device__ inline HeadTile split_tile(const TileSplit& s, int64_t v) {
    const int64_t hb = s.heads * s.body;
    if (v < hb) return HeadTile{static_cast<int>(v / s.body), v % s.body};
    const int64_t u = v - hb, tl = split_tail_len(s);
    return HeadTile{static_cast<int>(u / tl), s.body + u % tl};
}
// End of the run of virtual tiles that holds v and stays in one head's body or tail.
__host__ __device__ inline int64_t split_run_end(const TileSplit& s, int64_t v) {
    const int64_t hb = s.heads * s.body;
    if (v < hb) return (v / s.body + 1) * s.body;
    const int64_t tl = split_tail_len(s);
    return hb + ((v - hb) / tl + 1) * tl;
}
// Tail part that holds unit u of the concatenated tails (needs tail_chunks > 0).
__host__ __device__ inline int64_t split_tail_part(const TileSplit& s, int64_t u) {
    return ((u + 1) * s.tail_chunks - 1) / (s.heads * split_tail_len(s));
}

// split_tile in 32-bit arithmetic, for splits of fewer than 2^31 tiles.
__host__ __device__ inline void split_tile32(const TileSplit& s, int v, int& h, int& tile) {
    const int b = static_cast<int>(s.body), hb = s.heads * b;
    if (v < hb) {
        h = v / b;
        tile = v - h * b;
    } else {
        const int tl = static_cast<int>(s.tiles_per_head) - b, u = v - hb;
        h = u / tl;
        tile = b + (u - h * tl);
    }
}
// The apply kernels' schedules: no cap on the CTAs per head; a tail only where a CTA has
// at least 96 tiles (12288 tokens) of a head; a head switch in a tail part costs about 4
// tiles (its KV image is loaded and the pipeline refills).
constexpr int kNoPerHeadCap = 1 << 30;
constexpr int64_t kApplyMinPart = 96;
constexpr int64_t kApplySwitchCost = 4;

// Work chunks of the KV reduction: the split above of the layer's 64-token tiles over
// G = 152 chunks (one per SM of a 152-SM part) with k <= 150, a tail only where a chunk
// has at least 256 tiles (16384 tokens) of a head, and a head switch counted as 6 tiles
// (a partial written, the next head's first tiles refill the pipeline).  Each segment is summed by
// one CTA and leaves one partial KV: head h has k body partials (slots 0..k-1) and one or
// two tail partials (slots k, k+1).  The split is a function of (H, N) only, never read
// from the device, so the summation order is fixed by the shape.
constexpr int kChunks = 152;
constexpr int kChunksPerHeadCap = 150;  // k + 2 <= 152 keeps a head under kMaxSegments partials
constexpr int64_t kKvMinPart = 256;
constexpr int64_t kKvSwitchCost = 6;
constexpr int kMaxSegments = 160;       // partials per head the reduction can add

struct KvPlan : TileSplit {
    int seg_stride;  // partial slots per head: the most segments any head has
};

// Partial slot of (head h, chunk c) and the number of partials of head h.
__host__ __device__ inline int segment_of(const KvPlan& p, int h, int64_t c) {
    const int64_t kh = static_cast<int64_t>(p.per_head) * p.heads;
    if (c < kh) return static_cast<int>(c % p.per_head);
    const int64_t first = split_tail_part(p, static_cast<int64_t>(h) * split_tail_len(p));
    return p.per_head + static_cast<int>(c - kh - first);
}
__host__ __device__ inline int segments_of_head(const KvPlan& p, int h) {
    if (p.tail_chunks == 0) return p.per_head;
    const int64_t tl = split_tail_len(p);
    return p.per_head + static_cast<int>(split_tail_part(p, (h + 1) * tl - 1) - split_tail_part(p, h * tl) + 1);
}
__host__ __device__ inline KvPlan kv_plan(int heads, int64_t n_tokens) {
    KvPlan p;
    static_cast<TileSplit&>(p) = tile_split(heads, (n_tokens + kKvTile - 1) / kKvTile, kChunks, kChunksPerHeadCap,
                                            kKvMinPart, kKvSwitchCost);
    p.seg_stride = p.per_head;
    for (int h = 0; p.tail_chunks > 0 && h < heads; ++h) {
        const int n = segments_of_head(p, h);
        if (n > p.seg_stride) p.seg_stride = n;
    }
    return p;
}
// Largest seg_stride any n_tokens can produce for `heads` (scratch sizing): k is at most
// min(152 / H, 150), and a head's tail is never split more than twice (a tail part holds
// at least one head's whole tail, since E < H whenever k = floor(152 / H)).
__host__ __device__ inline int kv_seg_stride_bound(int heads) {
    const int k = tile_split(heads, kChunksPerHeadCap, kChunks, kChunksPerHeadCap, 0, 0).per_head;
    return k + (kChunks - k * heads > 0 ? 2 : 0);
}

// Work of one launch of the KV reduction: heads [h0, h0 + hc) of the layer (the K/V
// pointers and tensor maps start at head h0): their body chunks, then the tail chunks that
// touch them, each clipped to those heads.
struct KvLaunch {
    int h0;
    int n_body;                   // CTAs [0, n_body): body chunks c_body ...
    int n_chunks;                 // CTAs [n_body, n_chunks): tail chunks c_tail ...
    int64_t c_body, c_tail;
    int64_t tail_lo, tail_hi;     // virtual tiles of these heads' tails
};
__host__ __device__ inline KvLaunch kv_launch(const KvPlan& p, int h0, int hc) {
    KvLaunch l;
    l.h0 = h0;
    l.c_body = static_cast<int64_t>(h0) * p.per_head;
    l.n_body = hc * p.per_head;
    l.n_chunks = l.n_body;
    l.c_tail = l.tail_lo = l.tail_hi = 0;
    if (p.tail_chunks > 0) {
        const int64_t tl = split_tail_len(p), hb = p.heads * p.body;
        const int64_t e_lo = split_tail_part(p, h0 * tl), e_hi = split_tail_part(p, (h0 + hc) * tl - 1);
        l.c_tail = static_cast<int64_t>(p.per_head) * p.heads + e_lo;
        l.n_chunks += static_cast<int>(e_hi - e_lo + 1);
        l.tail_lo = hb + h0 * tl;
        l.tail_hi = hb + (h0 + hc) * tl;
    }
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
// With overlap = false the launch is an ordinary one: it starts only after everything
// before it in the stream (used where an event wait sits between two kernels and the second
// one reads what the waited-for work produced before its grid-dependency wait).
template <typename... Params, typename... Args>
cudaError_t launch_kernel(bool overlap, void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}
template <typename... Params, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
    return launch_kernel(true, kernel, grid, block, smem, stream, static_cast<Args&&>(args)...);
}

// The producer step fused into the tensor-core kernels (ReLU + interleaved RoPE on the
// loaded Q / K tiles, the normaliser from the activated un-rotated copies).
//   cos, sin : FP32 [N][D/2] rotation tables (pair p of token n is turned by cos/sin[n][p])
//   ksum_partial : FP64 [H][seg_stride][ksum_groups(D)][D] per-chunk, per-row-group column
//                  sums of relu(K) (scratch)
//   ksum : FP32 [H][D] reduced column sums (scratch; read by the apply)
// Row groups of the fused KV kernel's transform (one column-sum partial each): its 256
// threads are 16 chunk lanes x 16 row groups when the head dim spans two 64-column atoms,
// 8 lanes x 32 groups when it fits one.
__host__ __device__ constexpr int ksum_groups(int head_dim) { return head_dim <= 64 ? 32 : 16; }
constexpr int kKsumGroupsMax = 32;
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
    const __nv_bfloat162 zero2 = __float2bfloat162_rn(0.f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        // ReLU on the BF16 pair (one paired max; the same values as in binary32, a -0
        // input may come out as either zero), then each half widened exactly.
        const __nv_bfloat162 r = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&in[j]), zero2);
        const uint32_t rb = *reinterpret_cast<const uint32_t*>(&r);
        x0[j] = __uint_as_float(rb << 16);
        x1[j] = __uint_as_float(rb & 0xFFFF0000u);
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
// overlap = false: an ordinary launch (see launch_kernel).
cudaError_t launch_apply_tc(const CUtensorMap& tm_q, const CUtensorMap& tm_out, const uint8_t* kv_image,
                            const float* den, int heads, int64_t n_tokens, int head_dim, bool out_bf16,
                            bool token_major, int grid, int* status, uint64_t wait_ns, cudaStream_t stream,
                            bool overlap = true);

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
