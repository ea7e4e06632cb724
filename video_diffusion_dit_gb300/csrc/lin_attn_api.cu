// Host side of the lin_attn C ABI: argument checks, scratch ownership, TMA descriptors
// and the three-kernel enqueue per layer call.  See include/lin_attn.h for the contract.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>

#include "lin_attn.h"
#include "lin_attn_internal.cuh"

struct lin_attn_ctx {
    int device = 0;
    int heads = 0;
    int64_t max_tokens = 0;
    int head_dim = 0;
    int n_sms = 0;
    int seg_stride_alloc = 0;
    float* partial = nullptr;     // [heads][seg_stride_alloc][D][D] FP32 per-chunk partial sums
    float* kv = nullptr;          // [heads][D][D] FP32 reduced KV
    uint8_t* kv_image = nullptr;  // [heads] x three-term BF16 image for the tensor-core apply
    int* status = nullptr;        // device status word (LIN_ATTN_ERR_TIMEOUT if a kernel gave up)
    uint64_t wait_ns = la::kWaitLimitNs;  // how long a kernel waits on one of its barriers before giving up
    double* ksum_partial = nullptr;  // fused path: [heads][seg_stride_alloc][row groups][D] FP64 column sums of relu(K)
    float* ksum = nullptr;           // fused path: [heads][D] FP32 reduced column sums
    // host-buffer path staging, allocated on first use
    void* st_q = nullptr;
    void* st_k = nullptr;
    void* st_v = nullptr;
    float* st_den = nullptr;
    void* st_out = nullptr;
    float* st_cos = nullptr;  // fused host-buffer path: the rotation tables [max_tokens][D/2]
    float* st_sin = nullptr;
    // host-buffer pipeline: copy streams and ordering events, created on first use
    cudaStream_t s_in = nullptr;
    cudaStream_t s_out = nullptr;
    cudaEvent_t ev_ready = nullptr, ev_kv = nullptr, ev_in = nullptr, ev_comp = nullptr, ev_done = nullptr;
    // timing hook (one-shot)
    cudaEvent_t events[4] = {nullptr, nullptr, nullptr, nullptr};
    int n_events = 0;
};

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int ok() {
    g_last_error.clear();
    return LIN_ATTN_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(LIN_ATTN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Makes `device` current for the scope and restores the caller's device afterwards.
struct DeviceScope {
    int prev = -1;
    cudaError_t err = cudaSuccess;
    explicit DeviceScope(int device) {
        err = cudaGetDevice(&prev);
        if (err == cudaSuccess && prev != device) err = cudaSetDevice(device);
        else if (err == cudaSuccess) prev = -1;
    }
    ~DeviceScope() {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D map over a [.., N, .., D] activation of `h` heads with 128-byte swizzle; out-of-range
// elements read as zero and are skipped on stores.  Head-major ([H][N][D], `heads_total`
// unused): dims (D, N, H), box (box_x, rows, 1).  Token-major ([N][heads_total][D], the map
// covering `h` heads from `base`): dims (D, H, N), box (box_x, 1, rows).
// L2 promotion: a head-major tile is one contiguous run, fetched in 256-byte granules; a
// token-major tile is rows of D elements (224 bytes at D = 112) between other heads' rows,
// where 256-byte granules fetch the neighbours' bytes too, and they are mostly evicted again
// before the neighbour's CTA asks for them (22 % extra DRAM reads measured), so 64-byte
// granules for K and V; the apply's Q (and output) maps take 128-byte granules, which
// measured faster there (token-major apply 0.3916 -> 0.3787 ms at 720p, while K and V at
// 128 bytes made the KV kernel slower: 0.3062 -> 0.3152).
int make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, int64_t d, int64_t n,
             int64_t h, uint32_t box_x, uint32_t box_y, bool token_major = false, int64_t heads_total = 0,
             CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B,
             CUtensorMapL2promotion token_major_promotion = CU_TENSOR_MAP_L2_PROMOTION_L2_64B) {
    auto fn = encode_fn();
    if (!fn) return fail(LIN_ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(h)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d * elem_bytes), static_cast<cuuint64_t>(n * d * elem_bytes)};
    cuuint32_t box[3] = {box_x, box_y, 1};
    if (token_major) {
        dims[1] = static_cast<cuuint64_t>(h);
        dims[2] = static_cast<cuuint64_t>(n);
        strides[0] = static_cast<cuuint64_t>(d * elem_bytes);
        strides[1] = static_cast<cuuint64_t>(heads_total * d * elem_bytes);
        box[1] = 1;
        box[2] = box_y;
    }
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle, token_major ? token_major_promotion : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(LIN_ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return LIN_ATTN_OK;
}

// 2-D map over an FP32 [rows][cols] table (cols * 4 a multiple of 16), box (cols, box_rows),
// no swizzle: a box lands in shared memory as box_rows dense rows of cols floats.
int make_map_2d_f32(CUtensorMap* m, const float* base, int64_t cols, int64_t rows, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return fail(LIN_ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 4)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(cols), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(LIN_ATTN_ERR_CUDA, "cuTensorMapEncodeTiled (table) failed (CUresult %d)", (int)r);
    return LIN_ATTN_OK;
}

void free_all(lin_attn_ctx* c) {
    cudaFree(c->partial);
    cudaFree(c->kv);
    cudaFree(c->kv_image);
    cudaFree(c->status);
    cudaFree(c->ksum_partial);
    cudaFree(c->ksum);
    cudaFree(c->st_q);
    cudaFree(c->st_k);
    cudaFree(c->st_v);
    cudaFree(c->st_den);
    cudaFree(c->st_out);
    cudaFree(c->st_cos);
    cudaFree(c->st_sin);
    if (c->s_in) cudaStreamDestroy(c->s_in);
    if (c->s_out) cudaStreamDestroy(c->s_out);
    for (cudaEvent_t ev : {c->ev_ready, c->ev_kv, c->ev_in, c->ev_comp, c->ev_done})
        if (ev) cudaEventDestroy(ev);
}

int check_call(const lin_attn_ctx* ctx, const void* q, const void* k, const void* v, const float* den,
               const void* out, int out_dtype, int64_t n_tokens, int mode) {
    if (!ctx) return fail(LIN_ATTN_ERR_INVALID_ARG, "ctx is NULL");
    if (!q || !k || !v || !den || !out) return fail(LIN_ATTN_ERR_INVALID_ARG, "a tensor pointer is NULL");
    if (n_tokens < 1 || n_tokens > ctx->max_tokens)
        return fail(LIN_ATTN_ERR_INVALID_ARG, "n_tokens=%lld outside [1, %lld]", (long long)n_tokens,
                    (long long)ctx->max_tokens);
    if (mode != LIN_ATTN_MODE_HIGH && mode != LIN_ATTN_MODE_LOSSLESS)
        return fail(LIN_ATTN_ERR_INVALID_ARG, "mode=%d is not LIN_ATTN_MODE_HIGH/LOSSLESS", mode);
    if (out_dtype != LIN_ATTN_OUT_F32 && out_dtype != LIN_ATTN_OUT_BF16)
        return fail(LIN_ATTN_ERR_INVALID_ARG, "out_dtype=%d is not LIN_ATTN_OUT_F32/BF16", out_dtype);
    return LIN_ATTN_OK;
}

// Enqueue the three kernels for heads [h0, h0 + hc) of a layer whose tensors start at the
// given base pointers.  The split plan is always the one of the full head count, so a
// head range gives bitwise the same numbers as the whole layer.  `ev` (4 events or null)
// brackets the stages.
int enqueue_heads(lin_attn_ctx* c, const void* q, const void* k, const void* v, const float* den, void* out,
                  int out_dtype, int64_t n_tokens, int mode, cudaStream_t stream, int h0, int hc,
                  cudaEvent_t* ev, int layout = LIN_ATTN_LAYOUT_HND, const float* rope_cos = nullptr,
                  const float* rope_sin = nullptr, cudaEvent_t apply_after = nullptr) {
    const int H = c->heads, D = c->head_dim;
    const bool bf16_out = out_dtype == LIN_ATTN_OUT_BF16;
    const bool lossless = mode == LIN_ATTN_MODE_LOSSLESS;
    const bool tm = layout == LIN_ATTN_LAYOUT_NHD;  // token-major activations
    const la::KvPlan plan = la::kv_plan(H, n_tokens);
    const la::KvLaunch work = la::kv_launch(plan, h0, hc);
    const la::Strides sd = tm ? la::Strides{D, static_cast<int64_t>(H) * D}
                              : la::Strides{static_cast<int64_t>(n_tokens) * D, D};
    q = static_cast<const uint16_t*>(q) + h0 * sd.head;
    k = static_cast<const uint16_t*>(k) + h0 * sd.head;
    v = static_cast<const uint16_t*>(v) + h0 * sd.head;
    den += h0 * static_cast<size_t>(n_tokens);
    out = static_cast<uint8_t*>(out) + h0 * sd.head * (bf16_out ? 2 : 4);
    uint8_t* image_h0 = c->kv_image + h0 * static_cast<size_t>(la::kv_image_bytes(D));
    cudaError_t e;
    // Fused producer step: the KV kernel and the reduction index the column sums by layer
    // head, the apply by the launch's own heads.
    const bool fused = rope_cos != nullptr;
    const la::ProducerArgs pa_kv{rope_cos, rope_sin, c->ksum_partial, c->ksum, static_cast<int>(n_tokens)};
    const la::ProducerArgs pa_apply{rope_cos, rope_sin, c->ksum_partial, c->ksum + static_cast<size_t>(h0) * D,
                                    static_cast<int>(n_tokens)};

    if (ev && (e = cudaEventRecord(ev[0], stream)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    {
        CUtensorMap tk, tv;
        int rc = make_map(&tk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, n_tokens, hc, 64, la::kKvTile, tm, H);
        if (rc) return rc;
        rc = make_map(&tv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, n_tokens, hc, 64, la::kKvTile, tm, H);
        if (rc) return rc;
        CUtensorMap tabs[2];
        if (fused) {
            for (int t = 0; t < 2; ++t) {
                rc = make_map_2d_f32(&tabs[t], t ? rope_sin : rope_cos, D / 2, n_tokens, la::kKvTile);
                if (rc) return rc;
            }
        }
        e = la::launch_kv_partial_tc(tk, tv, c->partial, n_tokens, D, plan, work, tm, lossless, c->status, c->wait_ns,
                                     stream, fused ? &pa_kv : nullptr, fused ? tabs : nullptr);
        if (e != cudaSuccess) return cuda_fail(e, "kv_partial_tc launch");
    }
    if (ev && (e = cudaEventRecord(ev[1], stream)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    e = la::launch_kv_finalize(c->partial, c->kv, c->kv_image, h0, hc, D, plan, stream, fused ? &pa_kv : nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "kv_finalize launch");
    if (ev && (e = cudaEventRecord(ev[2], stream)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    // (host-buffer pipeline: Q and the denominators may still be on their way when the KV
    // kernels start; the apply, which fetches Q before its grid-dependency wait, is then
    // launched without the overlap so that it cannot start before they land)
    if (apply_after && (e = cudaStreamWaitEvent(stream, apply_after, 0)) != cudaSuccess)
        return cuda_fail(e, "stream ordering");
    {
        CUtensorMap tq, to;
        int rc = make_map(&tq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, n_tokens, hc, 64, la::kApplyTile, tm, H,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
        if (rc) return rc;
        if (fused) {  // transposed epilogue: (32 features, 32 tokens) boxes, unswizzled
            rc = bf16_out ? make_map(&to, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, n_tokens, hc, 32, 32, tm, H,
                                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B)
                          : make_map(&to, out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, n_tokens, hc, 32, 32, tm, H,
                                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
            if (rc) return rc;
            e = la::launch_apply_fused_tc(tq, to, image_h0, hc, n_tokens, D, bf16_out, tm, c->n_sms, c->status, c->wait_ns,
                                          stream, pa_apply);
        } else {
            rc = bf16_out ? make_map(&to, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, n_tokens, hc, 64, 32, tm, H,
                                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B)
                          : make_map(&to, out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, n_tokens, hc, 32, 32, tm, H,
                                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
            if (rc) return rc;
            e = la::launch_apply_tc(tq, to, image_h0, den, hc, n_tokens, D, bf16_out, tm, c->n_sms, c->status, c->wait_ns,
                                    stream, apply_after == nullptr);
        }
        if (e != cudaSuccess) return cuda_fail(e, "apply_tc launch");
    }
    if (ev && (e = cudaEventRecord(ev[3], stream)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    return ok();
}

// Heads per chunk of the host-buffer pipeline: about twenty chunks per layer (finer
// chunks expose less of the first upload and the last download; the kernels are cheap
// beside the copies).
constexpr int kHostChunks = 20;
int host_chunk_heads(int heads) { return heads >= kHostChunks ? (heads + kHostChunks - 1) / kHostChunks : 1; }

}  // namespace

namespace la {
// Sets the calling thread's last-error text (what lin_attn_last_error returns) for the
// library's other translation units; returns `code`.
int record_error(int code, const char* msg) {
    g_last_error = msg ? msg : "";
    return code;
}
}  // namespace la

extern "C" {

int lin_attn_version(void) { return LIN_ATTN_VERSION; }

const char* lin_attn_error_string(int status) {
    switch (status) {
        case LIN_ATTN_OK: return "ok";
        case LIN_ATTN_ERR_INVALID_ARG: return "invalid argument";
        case LIN_ATTN_ERR_UNSUPPORTED: return "unsupported shape or device";
        case LIN_ATTN_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
        case LIN_ATTN_ERR_CUDA: return "CUDA error";
        case LIN_ATTN_ERR_OOM: return "out of memory";
        case LIN_ATTN_ERR_TIMEOUT: return "kernel gave up waiting on a barrier";
        default: return "unknown status";
    }
}

const char* lin_attn_last_error(void) { return g_last_error.c_str(); }

int lin_attn_kv_plan(int heads, int64_t n_tokens, int mode, int* chunks, int* max_segments) {
    if (heads < 1 || n_tokens < 1 || (mode != LIN_ATTN_MODE_HIGH && mode != LIN_ATTN_MODE_LOSSLESS))
        return fail(LIN_ATTN_ERR_INVALID_ARG, "bad heads / n_tokens / mode");
    const la::KvPlan p = la::kv_plan(heads, n_tokens);
    int most = 0;
    for (int h = 0; h < heads; ++h) {
        const int n = la::segments_of_head(p, h);
        most = n > most ? n : most;
    }
    if (chunks) *chunks = p.chunks;
    if (max_segments) *max_segments = most;
    return ok();
}

int lin_attn_create(lin_attn_ctx** out_ctx, int heads, int64_t max_tokens, int head_dim, int device) {
    if (!out_ctx) return fail(LIN_ATTN_ERR_INVALID_ARG, "ctx out-pointer is NULL");
    *out_ctx = nullptr;
    if (heads < 1 || heads > 4096) return fail(LIN_ATTN_ERR_INVALID_ARG, "heads=%d outside [1, 4096]", heads);
    if (max_tokens < 1 || max_tokens > (int64_t(1) << 30))
        return fail(LIN_ATTN_ERR_INVALID_ARG, "max_tokens=%lld outside [1, 2^30]", (long long)max_tokens);
    if (head_dim < 16 || head_dim > 128 || head_dim % 16 != 0)
        return fail(LIN_ATTN_ERR_UNSUPPORTED, "head_dim=%d is not a multiple of 16 in [16, 128]", head_dim);
    if (static_cast<int64_t>(heads) * max_tokens > (int64_t(1) << 31) - 1)
        return fail(LIN_ATTN_ERR_INVALID_ARG, "heads * max_tokens exceeds 2^31 - 1");
    int count = 0;
    cudaError_t e = cudaGetDeviceCount(&count);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
    if (device < 0 || device >= count)
        return fail(LIN_ATTN_ERR_INVALID_ARG, "device=%d outside [0, %d)", device, count);
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (major != 10 || minor != 3)
        return fail(LIN_ATTN_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", device,
                    major, minor);
    DeviceScope scope(device);
    if (scope.err != cudaSuccess) return cuda_fail(scope.err, "cudaSetDevice");

    auto* c = new lin_attn_ctx();
    c->device = device;
    c->heads = heads;
    c->max_tokens = max_tokens;
    c->head_dim = head_dim;
    c->n_sms = sms;
    c->seg_stride_alloc = la::kv_seg_stride_bound(heads);
    const size_t dd = static_cast<size_t>(head_dim) * head_dim;
    bool good = cudaMalloc(&c->partial, sizeof(float) * dd * heads * c->seg_stride_alloc) == cudaSuccess &&
                cudaMalloc(&c->kv, sizeof(float) * dd * heads) == cudaSuccess &&
                cudaMalloc(&c->kv_image, static_cast<size_t>(la::kv_image_bytes(head_dim)) * heads) == cudaSuccess &&
                cudaMalloc(&c->status, sizeof(int)) == cudaSuccess &&
                cudaMalloc(&c->ksum_partial, sizeof(double) * heads * c->seg_stride_alloc * la::kKsumGroupsMax * head_dim) ==
                    cudaSuccess &&
                cudaMalloc(&c->ksum, sizeof(float) * heads * head_dim) == cudaSuccess;
    if (!good) {
        cudaGetLastError();
        free_all(c);
        delete c;
        return fail(LIN_ATTN_ERR_OOM, "device allocation of the context scratch failed");
    }
    // The image's padding columns (head-dim index >= D inside the last 64-column atom) stay zero.
    if ((e = cudaMemset(c->kv_image, 0, static_cast<size_t>(la::kv_image_bytes(head_dim)) * heads)) != cudaSuccess ||
        (e = cudaMemset(c->status, 0, sizeof(int))) != cudaSuccess ||
        (e = cudaDeviceSynchronize()) != cudaSuccess) {
        free_all(c);
        delete c;
        return cuda_fail(e, "context initialisation");
    }
    *out_ctx = c;
    return ok();
}

int lin_attn_destroy(lin_attn_ctx* ctx) {
    if (!ctx) return ok();
    DeviceScope scope(ctx->device);
    if (scope.err == cudaSuccess) cudaDeviceSynchronize();
    free_all(ctx);
    delete ctx;
    return ok();
}

int lin_attn_forward(lin_attn_ctx* ctx, const void* q_rot, const void* k_rot, const void* v, const float* normalizer,
                     void* out, int out_dtype, int64_t n_tokens, int mode, struct CUstream_st* stream) {
    int rc = check_call(ctx, q_rot, k_rot, v, normalizer, out, out_dtype, n_tokens, mode);
    if (rc) return rc;
    if (!aligned16(q_rot) || !aligned16(k_rot) || !aligned16(v) || !aligned16(normalizer) || !aligned16(out))
        return fail(LIN_ATTN_ERR_MISALIGNED, "every tensor pointer must be 16-byte aligned");
    DeviceScope scope(ctx->device);
    if (scope.err != cudaSuccess) return cuda_fail(scope.err, "cudaSetDevice");
    cudaEvent_t* ev = ctx->n_events == 4 ? ctx->events : nullptr;
    ctx->n_events = 0;
    return enqueue_heads(ctx, q_rot, k_rot, v, normalizer, out, out_dtype, n_tokens, mode,
                         reinterpret_cast<cudaStream_t>(stream), 0, ctx->heads, ev);
}

int lin_attn_forward_layout(lin_attn_ctx* ctx, const void* q_rot, const void* k_rot, const void* v,
                            const float* normalizer, void* out, int out_dtype, int64_t n_tokens, int mode, int layout,
                            struct CUstream_st* stream) {
    int rc = check_call(ctx, q_rot, k_rot, v, normalizer, out, out_dtype, n_tokens, mode);
    if (rc) return rc;
    if (layout != LIN_ATTN_LAYOUT_HND && layout != LIN_ATTN_LAYOUT_NHD)
        return fail(LIN_ATTN_ERR_INVALID_ARG, "layout=%d is not LIN_ATTN_LAYOUT_HND/NHD", layout);
    if (!aligned16(q_rot) || !aligned16(k_rot) || !aligned16(v) || !aligned16(normalizer) || !aligned16(out))
        return fail(LIN_ATTN_ERR_MISALIGNED, "every tensor pointer must be 16-byte aligned");
    DeviceScope scope(ctx->device);
    if (scope.err != cudaSuccess) return cuda_fail(scope.err, "cudaSetDevice");
    cudaEvent_t* ev = ctx->n_events == 4 ? ctx->events : nullptr;
    ctx->n_events = 0;
    return enqueue_heads(ctx, q_rot, k_rot, v, normalizer, out, out_dtype, n_tokens, mode,
                         reinterpret_cast<cudaStream_t>(stream), 0, ctx->heads, ev, layout);
}

int lin_attn_forward_fused(lin_attn_ctx* ctx, const void* q, const void* k, const void* v, const float* rope_cos,
                           const float* rope_sin, void* out, int out_dtype, int64_t n_tokens, int mode,
                           struct CUstream_st* stream) {
    return lin_attn_forward_fused_layout(ctx, q, k, v, rope_cos, rope_sin, out, out_dtype, n_tokens, mode,
                                         LIN_ATTN_LAYOUT_HND, stream);
}

int lin_attn_forward_fused_layout(lin_attn_ctx* ctx, const void* q, const void* k, const void* v,
                                  const float* rope_cos, const float* rope_sin, void* out, int out_dtype,
                                  int64_t n_tokens, int mode, int layout, struct CUstream_st* stream) {
    if (layout != LIN_ATTN_LAYOUT_HND && layout != LIN_ATTN_LAYOUT_NHD)
        return fail(LIN_ATTN_ERR_INVALID_ARG, "layout=%d is not LIN_ATTN_LAYOUT_HND/NHD", layout);
    if (!rope_cos || !rope_sin) return fail(LIN_ATTN_ERR_INVALID_ARG, "rotation table pointer is NULL");
    // check_call wants a denominator pointer; the fused call forms the denominators itself.
    int rc = check_call(ctx, q, k, v, rope_cos, out, out_dtype, n_tokens, mode);
    if (rc) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(rope_cos) || !aligned16(rope_sin) ||
        !aligned16(out))
        return fail(LIN_ATTN_ERR_MISALIGNED, "every tensor pointer must be 16-byte aligned");
    DeviceScope scope(ctx->device);
    if (scope.err != cudaSuccess) return cuda_fail(scope.err, "cudaSetDevice");
    cudaEvent_t* ev = ctx->n_events == 4 ? ctx->events : nullptr;
    ctx->n_events = 0;
    return enqueue_heads(ctx, q, k, v, nullptr, out, out_dtype, n_tokens, mode, reinterpret_cast<cudaStream_t>(stream),
                         0, ctx->heads, ev, layout, rope_cos, rope_sin);
}

int lin_attn_anchor_forward(lin_attn_ctx* ctx, const void* q, const void* k, const void* v, void* out,
                            int out_dtype, int64_t n_tokens, float scale, struct CUstream_st* stream) {
    if (!ctx) return fail(LIN_ATTN_ERR_INVALID_ARG, "ctx is NULL");
    if (!q || !k || !v || !out) return fail(LIN_ATTN_ERR_INVALID_ARG, "a tensor pointer is NULL");
    if (n_tokens < 1 || n_tokens > ctx->max_tokens)
        return fail(LIN_ATTN_ERR_INVALID_ARG, "n_tokens=%lld outside [1, %lld]", (long long)n_tokens,
                    (long long)ctx->max_tokens);
    if (out_dtype != LIN_ATTN_OUT_F32 && out_dtype != LIN_ATTN_OUT_BF16)
        return fail(LIN_ATTN_ERR_INVALID_ARG, "out_dtype=%d is not LIN_ATTN_OUT_F32/BF16", out_dtype);
    if (!(scale >= 0.0f) || !(scale < 1e30f)) return fail(LIN_ATTN_ERR_INVALID_ARG, "scale must be finite and >= 0");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return fail(LIN_ATTN_ERR_MISALIGNED, "every tensor pointer must be 16-byte aligned");
    DeviceScope scope(ctx->device);
    if (scope.err != cudaSuccess) return cuda_fail(scope.err, "cudaSetDevice");
    const int H = ctx->heads, D = ctx->head_dim;
    const float s = scale > 0.0f ? scale : 1.0f / sqrtf(static_cast<float>(D));
    const float log2e = 1.4426950408889634f;
    CUtensorMap tq, tk, tv;
    int rc = make_map(&tq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, n_tokens, H, 64, 128);
    if (rc) return rc;
    if ((rc = make_map(&tk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, n_tokens, H, 64, 128))) return rc;
    if ((rc = make_map(&tv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, n_tokens, H, 64, 128))) return rc;
    cudaError_t e = la::launch_anchor_attention(tq, tk, tv, out, out_dtype == LIN_ATTN_OUT_BF16, H, n_tokens, D,
                                                s * log2e, ctx->status, ctx->wait_ns,
                                                reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "anchor_attention launch");
    return ok();
}

namespace {

// The host-buffer pipeline shared by the plain and the fused call.  den is the plain call's
// denominators; rope_cos / rope_sin (both or neither) make it the fused call, whose tables
// are copied once, ahead of the first chunk's K and V.
int host_pipeline(lin_attn_ctx* ctx, const void* q, const void* k, const void* v, const float* den,
                  const float* rope_cos, const float* rope_sin, void* out, int out_dtype, int64_t n_tokens, int mode,
                  cudaStream_t s) {
    DeviceScope scope(ctx->device);
    if (scope.err != cudaSuccess) return cuda_fail(scope.err, "cudaSetDevice");
    const bool fused = rope_cos != nullptr;
    const size_t elems_max = static_cast<size_t>(ctx->heads) * ctx->max_tokens * ctx->head_dim;
    if (!ctx->st_q) {
        bool good = cudaMalloc(&ctx->st_q, 2 * elems_max) == cudaSuccess &&
                    cudaMalloc(&ctx->st_k, 2 * elems_max) == cudaSuccess &&
                    cudaMalloc(&ctx->st_v, 2 * elems_max) == cudaSuccess &&
                    cudaMalloc(&ctx->st_den, 4 * static_cast<size_t>(ctx->heads) * ctx->max_tokens) == cudaSuccess &&
                    cudaMalloc(&ctx->st_out, 4 * elems_max) == cudaSuccess;
        if (!good) {
            cudaGetLastError();
            cudaFree(ctx->st_q);
            cudaFree(ctx->st_k);
            cudaFree(ctx->st_v);
            cudaFree(ctx->st_den);
            cudaFree(ctx->st_out);
            ctx->st_q = ctx->st_k = ctx->st_v = ctx->st_out = nullptr;
            ctx->st_den = nullptr;
            return fail(LIN_ATTN_ERR_OOM, "device allocation of the host-path staging failed");
        }
    }
    const size_t table_bytes = static_cast<size_t>(n_tokens) * (ctx->head_dim / 2) * sizeof(float);
    if (fused && !ctx->st_cos) {
        const size_t max_bytes = static_cast<size_t>(ctx->max_tokens) * (ctx->head_dim / 2) * sizeof(float);
        if (cudaMalloc(&ctx->st_cos, max_bytes) != cudaSuccess || cudaMalloc(&ctx->st_sin, max_bytes) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(ctx->st_cos);
            cudaFree(ctx->st_sin);
            ctx->st_cos = ctx->st_sin = nullptr;
            return fail(LIN_ATTN_ERR_OOM, "device allocation of the host-path table staging failed");
        }
    }
    cudaError_t e;
    if (!ctx->s_in) {
        if ((e = cudaStreamCreateWithFlags(&ctx->s_in, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&ctx->s_out, cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_fail(e, "cudaStreamCreate");
        for (cudaEvent_t* ev : {&ctx->ev_ready, &ctx->ev_kv, &ctx->ev_in, &ctx->ev_comp, &ctx->ev_done})
            if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail(e, "cudaEventCreate");
    }
    // Pipeline over chunks of heads: host-to-device copies on one stream, the kernels on
    // the caller's stream, device-to-host copies on a third, so both copy directions and
    // the compute overlap.  Each chunk waits only for its own inputs.
    const int H = ctx->heads, chunk = host_chunk_heads(H);
    const size_t head_elems = static_cast<size_t>(n_tokens) * ctx->head_dim;
    const size_t out_es = out_dtype == LIN_ATTN_OUT_BF16 ? 2 : 4;
    auto hptr = [](const void* p, size_t off) { return static_cast<const uint8_t*>(p) + off; };
    auto dptr = [](void* p, size_t off) { return static_cast<uint8_t*>(p) + off; };
    if ((e = cudaEventRecord(ctx->ev_ready, s)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(ctx->s_in, ctx->ev_ready, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(ctx->s_out, ctx->ev_ready, 0)) != cudaSuccess)
        return cuda_fail(e, "stream ordering");
    if (fused && ((e = cudaMemcpyAsync(ctx->st_cos, rope_cos, table_bytes, cudaMemcpyHostToDevice, ctx->s_in)) !=
                      cudaSuccess ||
                  (e = cudaMemcpyAsync(ctx->st_sin, rope_sin, table_bytes, cudaMemcpyHostToDevice, ctx->s_in)) !=
                      cudaSuccess))
        return cuda_fail(e, "host-to-device copy");
    for (int h0 = 0; h0 < H; h0 += chunk) {
        const int hc = h0 + chunk <= H ? chunk : H - h0;
        const size_t off = h0 * head_elems * 2, bytes = hc * head_elems * 2;
        const size_t doff = h0 * static_cast<size_t>(n_tokens) * 4, dbytes = hc * static_cast<size_t>(n_tokens) * 4;
        // K and V first (and, on the fused path, the tables before the first chunk): the
        // chunk's KV kernels wait only for them, the apply also for Q (and the denominators),
        // which are copied while the KV kernels run.
        if ((e = cudaMemcpyAsync(dptr(ctx->st_k, off), hptr(k, off), bytes, cudaMemcpyHostToDevice, ctx->s_in)) !=
                cudaSuccess ||
            (e = cudaMemcpyAsync(dptr(ctx->st_v, off), hptr(v, off), bytes, cudaMemcpyHostToDevice, ctx->s_in)) !=
                cudaSuccess)
            return cuda_fail(e, "host-to-device copy");
        if ((e = cudaEventRecord(ctx->ev_kv, ctx->s_in)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(s, ctx->ev_kv, 0)) != cudaSuccess)
            return cuda_fail(e, "stream ordering");
        if ((e = cudaMemcpyAsync(dptr(ctx->st_q, off), hptr(q, off), bytes, cudaMemcpyHostToDevice, ctx->s_in)) !=
            cudaSuccess)
            return cuda_fail(e, "host-to-device copy");
        if (!fused && (e = cudaMemcpyAsync(dptr(ctx->st_den, doff), hptr(den, doff), dbytes, cudaMemcpyHostToDevice,
                                           ctx->s_in)) != cudaSuccess)
            return cuda_fail(e, "host-to-device copy");
        if ((e = cudaEventRecord(ctx->ev_in, ctx->s_in)) != cudaSuccess) return cuda_fail(e, "stream ordering");
        const int rc = enqueue_heads(ctx, ctx->st_q, ctx->st_k, ctx->st_v, fused ? nullptr : ctx->st_den, ctx->st_out,
                                     out_dtype, n_tokens, mode, s, h0, hc, nullptr, LIN_ATTN_LAYOUT_HND,
                                     fused ? ctx->st_cos : nullptr, fused ? ctx->st_sin : nullptr, ctx->ev_in);
        if (rc) return rc;
        if ((e = cudaEventRecord(ctx->ev_comp, s)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(ctx->s_out, ctx->ev_comp, 0)) != cudaSuccess)
            return cuda_fail(e, "stream ordering");
        const size_t ooff = h0 * head_elems * out_es, obytes = hc * head_elems * out_es;
        if ((e = cudaMemcpyAsync(dptr(out, ooff), dptr(ctx->st_out, ooff), obytes, cudaMemcpyDeviceToHost,
                                 ctx->s_out)) != cudaSuccess)
            return cuda_fail(e, "device-to-host copy");
    }
    if ((e = cudaEventRecord(ctx->ev_done, ctx->s_out)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s, ctx->ev_done, 0)) != cudaSuccess)
        return cuda_fail(e, "stream ordering");
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    return ok();
}

}  // namespace

int lin_attn_forward_host(lin_attn_ctx* ctx, const void* q_rot, const void* k_rot, const void* v,
                          const float* normalizer, void* out, int out_dtype, int64_t n_tokens, int mode,
                          struct CUstream_st* stream) {
    const int rc = check_call(ctx, q_rot, k_rot, v, normalizer, out, out_dtype, n_tokens, mode);
    if (rc) return rc;
    return host_pipeline(ctx, q_rot, k_rot, v, normalizer, nullptr, nullptr, out, out_dtype, n_tokens, mode,
                         reinterpret_cast<cudaStream_t>(stream));
}

int lin_attn_forward_fused_host(lin_attn_ctx* ctx, const void* q, const void* k, const void* v, const float* rope_cos,
                                const float* rope_sin, void* out, int out_dtype, int64_t n_tokens, int mode,
                                struct CUstream_st* stream) {
    if (!rope_cos || !rope_sin) return fail(LIN_ATTN_ERR_INVALID_ARG, "rotation table pointer is NULL");
    // check_call wants a denominator pointer; the fused call forms the denominators itself.
    const int rc = check_call(ctx, q, k, v, rope_cos, out, out_dtype, n_tokens, mode);
    if (rc) return rc;
    return host_pipeline(ctx, q, k, v, nullptr, rope_cos, rope_sin, out, out_dtype, n_tokens, mode,
                         reinterpret_cast<cudaStream_t>(stream));
}

int lin_attn_debug_kv(lin_attn_ctx* ctx, float* kv_out, struct CUstream_st* stream) {
    if (!ctx || !kv_out) return fail(LIN_ATTN_ERR_INVALID_ARG, "ctx or kv_out is NULL");
    DeviceScope scope(ctx->device);
    if (scope.err != cudaSuccess) return cuda_fail(scope.err, "cudaSetDevice");
    const size_t bytes = sizeof(float) * ctx->heads * static_cast<size_t>(ctx->head_dim) * ctx->head_dim;
    cudaError_t e = cudaMemcpyAsync(kv_out, ctx->kv, bytes, cudaMemcpyDeviceToDevice,
                                    reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "debug_kv copy");
    return ok();
}

int lin_attn_device_status(lin_attn_ctx* ctx, struct CUstream_st* stream) {
    if (!ctx) return fail(LIN_ATTN_ERR_INVALID_ARG, "ctx is NULL");
    DeviceScope scope(ctx->device);
    if (scope.err != cudaSuccess) return cuda_fail(scope.err, "cudaSetDevice");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int h = 0;
    if ((e = cudaMemcpy(&h, ctx->status, sizeof h, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "status read");
    if (h != 0) {
        cudaMemset(ctx->status, 0, sizeof(int));
        return fail(h, "a kernel reported status %d (%s)", h, lin_attn_error_string(h));
    }
    return ok();
}

int lin_attn_set_wait_limit(lin_attn_ctx* ctx, uint64_t limit_ns) {
    if (!ctx) return fail(LIN_ATTN_ERR_INVALID_ARG, "ctx is NULL");
    if (limit_ns > la::kWaitLimitNs)
        return fail(LIN_ATTN_ERR_INVALID_ARG, "limit_ns=%llu exceeds the default %llu", (unsigned long long)limit_ns,
                    (unsigned long long)la::kWaitLimitNs);
    ctx->wait_ns = limit_ns == 0 ? la::kWaitLimitNs : limit_ns;
    return ok();
}

int lin_attn_set_stage_events(lin_attn_ctx* ctx, struct CUevent_st* const* events, int n_events) {
    if (!ctx) return fail(LIN_ATTN_ERR_INVALID_ARG, "ctx is NULL");
    if (n_events == 0) {
        ctx->n_events = 0;
        return ok();
    }
    if (n_events != 4 || !events) return fail(LIN_ATTN_ERR_INVALID_ARG, "n_events must be 4 (or 0 to disarm)");
    for (int i = 0; i < 4; ++i) {
        if (!events[i]) return fail(LIN_ATTN_ERR_INVALID_ARG, "event %d is NULL", i);
        ctx->events[i] = reinterpret_cast<cudaEvent_t>(events[i]);
    }
    ctx->n_events = 4;
    return ok();
}

}  // extern "C"
