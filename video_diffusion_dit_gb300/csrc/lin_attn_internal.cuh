// Shared declarations of the lin_attn kernels and their host-side launchers.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace la {

// Token tile of the tensor-core KV partial kernel (rows per pipeline stage).
constexpr int kKvTile = 64;
// Token tile of the tensor-core apply kernel (MMA M).
constexpr int kApplyTile = 128;
// Upper bound on token splits per head (the reduction keeps one FP32 value per split in
// registers).
constexpr int kMaxSplits = 64;
// Target number of (head, split) work units of the KV partial kernel: a constant chosen
// for a 152-SM part, so the split plan - and with it the summation order - is fixed by
// the shape alone.
constexpr int kSplitUnitsTarget = 760;

struct SplitPlan {
    int splits;     // S: splits per head
    int64_t chunk;  // tokens per split (multiple of kKvTile); the last split may be shorter
};

__host__ __device__ inline SplitPlan split_plan(int heads, int64_t n_tokens) {
    int s0 = (kSplitUnitsTarget + heads - 1) / heads;
    if (s0 < 1) s0 = 1;
    if (s0 > kMaxSplits) s0 = kMaxSplits;
    int64_t per = (n_tokens + s0 - 1) / s0;
    int64_t chunk = ((per + kKvTile - 1) / kKvTile) * kKvTile;
    if (chunk < kKvTile) chunk = kKvTile;
    SplitPlan p;
    p.chunk = chunk;
    p.splits = static_cast<int>((n_tokens + chunk - 1) / chunk);
    return p;
}

// Number of 64-wide column blocks ("atoms") that cover the head dim: 1 for D <= 64, else 2.
__host__ __device__ inline int head_dim_atoms(int head_dim) { return (head_dim + 63) / 64; }

// Bytes of one head's three-term BF16 image of KV^T in the 128-byte-swizzled K-major
// layout the apply kernel's MMA reads straight from shared memory.
__host__ __device__ inline int64_t kv_image_bytes(int head_dim) {
    return 3ll * head_dim_atoms(head_dim) * head_dim * 128;
}

// Sets the calling thread's last-error text (lin_attn_last_error); returns `code`.
int record_error(int code, const char* msg);

// ---------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error.

// KV partial sums on tensor cores (BF16 x BF16 -> FP32): partial[h][s][i][j].
cudaError_t launch_kv_partial_tc(const CUtensorMap& tm_k, const CUtensorMap& tm_v, float* partial, int heads,
                                 int64_t n_tokens, int head_dim, SplitPlan plan, int grid, int* status,
                                 cudaStream_t stream);

// KV partial sums with FP32 FMA on CUDA cores (operands upcast from BF16).
cudaError_t launch_kv_partial_ffma(const uint16_t* k, const uint16_t* v, float* partial, int heads,
                                   int64_t n_tokens, int head_dim, SplitPlan plan, cudaStream_t stream);

// Fixed-order pairwise reduction of the split partials: kv[h][i][j] (FP32) and, if
// kv_image != nullptr, its three-term BF16 image for the tensor-core apply.
cudaError_t launch_kv_finalize(const float* partial, float* kv, uint8_t* kv_image, int heads, int head_dim,
                               int splits, cudaStream_t stream);

// out = (Q . KV) * (1 / den) on tensor cores, KV as three BF16 terms.
cudaError_t launch_apply_tc(const CUtensorMap& tm_q, const CUtensorMap& tm_out, const uint8_t* kv_image,
                            const float* den, int heads, int64_t n_tokens, int head_dim, bool out_bf16, int grid,
                            int* status, cudaStream_t stream);

// out = (Q . KV) * (1 / den) with FP32 FMA on CUDA cores.
cudaError_t launch_apply_ffma(const uint16_t* q, const float* kv, const float* den, void* out, int heads,
                              int64_t n_tokens, int head_dim, bool out_bf16, int grid, cudaStream_t stream);

}  // namespace la
