// lin_attn_forward_noalloc: the layer call for callers that cannot allocate device memory.
//
// The regular entry point keeps its scratch (per-chunk KV partial sums, the reduced KV,
// the KV image the apply kernel reads, a status word) in a context made by
// lin_attn_create, which calls cudaMalloc.  Some callers cannot do that: a plugin whose
// host forbids allocation inside its enqueue/execute callback, a serving process whose
// device memory is entirely reserved up front by a caching allocator or a memory cap, or
// a latency-critical loop that must not hit cudaMalloc's implicit device synchronisation.
// This entry point serves them from one fixed scratch array compiled into the library:
// it calls no cudaMalloc, cudaFree or allocating library routine.
//
// The array (kNoAllocScratchBytes) is a file-scope __device__ variable, so every GPU that
// loads this library holds it until the process exits.  Its host-side name is only a
// stand-in for the symbol, never a device address: the first call on each device (with
// that device current) resolves the real address with cudaGetSymbolAddress and caches it
// (a failed attempt is not cached; the next call retries), and that first call should
// therefore come before any stream capture.  All
// calls share the array and it keeps the previous call's contents: the parts that must
// start at zero are cleared by every call, and calls whose execution overlaps on the GPU
// (two streams, or two host threads) race on it and give wrong results.  Its first 256
// bytes hold the status word, where a kernel that gave up waiting records the timeout;
// lin_attn_noalloc_status reads and clears it.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "lin_attn.h"
#include "lin_attn_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(48) << 20;  // 48 MiB
constexpr int kMaxDevices = 64;
constexpr size_t kStatusBytes = 256;  // the status word's slot at the start of the scratch

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Per-device set-up.  Only a successful set-up is kept: if resolving the address fails
// (for instance because the first call was made while a stream was being captured), the
// next call on that device tries again.
struct DeviceSetup {
    bool resolved = false;
    unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int n_sms = 0;
    bool supported = false;
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mutex;

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

// Same 3-D [H][N][D] map (128-byte swizzle, zero fill) as the context path uses.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, int64_t d, int64_t n,
              int64_t h, uint32_t box_x, uint32_t box_y) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(h)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d * elem_bytes), static_cast<cuuint64_t>(n * d * elem_bytes)};
    cuuint32_t box[3] = {box_x, box_y, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    return la::record_error(code, buf);
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(LIN_ATTN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// The calling thread's current device's set-up, resolved on first use (see DeviceSetup).
int device_setup(DeviceSetup* out) {
    int device = -1;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (device < 0 || device >= kMaxDevices) return fail(LIN_ATTN_ERR_UNSUPPORTED, "device index %d too large", device);
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    DeviceSetup& slot = g_setup[device];
    if (!slot.resolved) {
        int major = 0, minor = 0, sms = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (major != 10 || minor != 3) return fail(LIN_ATTN_ERR_UNSUPPORTED, "device %d is not sm_103", device);
        unsigned char* addr = nullptr;
        e = cudaGetSymbolAddress(reinterpret_cast<void**>(&addr), g_noalloc_scratch);
        if (e != cudaSuccess || !addr) {
            cudaGetLastError();  // not sticky; leave the set-up open for the next call
            return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
        }
        slot.scratch = addr;
        slot.n_sms = sms;
        slot.supported = true;
        slot.resolved = true;
    }
    *out = slot;
    return LIN_ATTN_OK;
}

}  // namespace

extern "C" int lin_attn_forward_noalloc(const void* q_rot, const void* k_rot, const void* v,
                                        const float* normalizer, void* out, int out_dtype, int heads,
                                        int64_t n_tokens, int head_dim, int mode, struct CUstream_st* stream) {
    if (!q_rot || !k_rot || !v || !normalizer || !out) return fail(LIN_ATTN_ERR_INVALID_ARG, "a tensor pointer is NULL");
    if (heads < 1 || heads > 4096) return fail(LIN_ATTN_ERR_INVALID_ARG, "heads=%d outside [1, 4096]", heads);
    if (n_tokens < 1 || n_tokens > (int64_t(1) << 30) || static_cast<int64_t>(heads) * n_tokens > (int64_t(1) << 31) - 1)
        return fail(LIN_ATTN_ERR_INVALID_ARG, "n_tokens=%lld out of range", (long long)n_tokens);
    if (head_dim < 16 || head_dim > 128 || head_dim % 16 != 0)
        return fail(LIN_ATTN_ERR_UNSUPPORTED, "head_dim=%d is not a multiple of 16 in [16, 128]", head_dim);
    if (mode != LIN_ATTN_MODE_HIGH && mode != LIN_ATTN_MODE_LOSSLESS)
        return fail(LIN_ATTN_ERR_INVALID_ARG, "mode=%d is not LIN_ATTN_MODE_HIGH/LOSSLESS", mode);
    if (out_dtype != LIN_ATTN_OUT_F32 && out_dtype != LIN_ATTN_OUT_BF16)
        return fail(LIN_ATTN_ERR_INVALID_ARG, "out_dtype=%d is not LIN_ATTN_OUT_F32/BF16", out_dtype);
    for (const void* p : {q_rot, k_rot, v, static_cast<const void*>(normalizer), static_cast<const void*>(out)})
        if (reinterpret_cast<uintptr_t>(p) & 15u)
            return fail(LIN_ATTN_ERR_MISALIGNED, "every tensor pointer must be 16-byte aligned");

    // Scratch carve-up: status word | partials | KV | KV image, each 256-byte aligned.  The
    // status word sits at a fixed place so that lin_attn_noalloc_status can find it.
    const la::KvPlan plan = la::kv_plan(heads, n_tokens);
    const la::KvLaunch work = la::kv_launch(plan, 0, heads);
    const size_t dd = static_cast<size_t>(head_dim) * head_dim;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t partial_bytes = up(sizeof(float) * dd * heads * plan.seg_stride);
    const size_t kv_bytes = up(sizeof(float) * dd * heads);
    const size_t image_bytes = static_cast<size_t>(la::kv_image_bytes(head_dim)) * heads;
    const size_t need = kStatusBytes + partial_bytes + kv_bytes + up(image_bytes);
    if (need > kNoAllocScratchBytes)
        return fail(LIN_ATTN_ERR_INVALID_ARG,
                    "this shape needs %zu bytes of scratch, more than the %zu built into the library for "
                    "lin_attn_forward_noalloc; use a context (lin_attn_create) instead",
                    need, kNoAllocScratchBytes);

    DeviceSetup su;
    if (const int rc = device_setup(&su)) return rc;
    cudaError_t e;

    int* status = reinterpret_cast<int*>(su.scratch);
    float* partial = reinterpret_cast<float*>(su.scratch + kStatusBytes);
    float* kv = reinterpret_cast<float*>(su.scratch + kStatusBytes + partial_bytes);
    uint8_t* image = su.scratch + kStatusBytes + partial_bytes + kv_bytes;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool bf16_out = out_dtype == LIN_ATTN_OUT_BF16;

    // Must start at zero: the KV image (its padding columns are read by the MMA and a
    // previous call with another head dim may have left data there).  The status word is
    // not cleared here: it collects timeouts until lin_attn_noalloc_status reads it.
    if ((e = cudaMemsetAsync(image, 0, image_bytes, s)) != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");

    CUtensorMap tk, tv;
    if (!make_map(&tk, k_rot, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, head_dim, n_tokens, heads, 64, la::kKvTile) ||
        !make_map(&tv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, head_dim, n_tokens, heads, 64, la::kKvTile))
        return fail(LIN_ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    e = la::launch_kv_partial_tc(tk, tv, partial, n_tokens, head_dim, plan, work, false, mode == LIN_ATTN_MODE_LOSSLESS,
                                 status, la::kWaitLimitNs, s);
    if (e != cudaSuccess) return cuda_fail(e, "kv_partial launch");
    e = la::launch_kv_finalize(partial, kv, image, 0, heads, head_dim, plan, s);
    if (e != cudaSuccess) return cuda_fail(e, "kv_finalize launch");
    CUtensorMap tq, to;
    const bool okq = make_map(&tq, q_rot, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, head_dim, n_tokens, heads, 64,
                              la::kApplyTile);
    const bool oko = bf16_out ? make_map(&to, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, head_dim, n_tokens, heads, 64, 32)
                              : make_map(&to, out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, head_dim, n_tokens, heads, 32, 32);
    if (!okq || !oko) return fail(LIN_ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    e = la::launch_apply_tc(tq, to, image, normalizer, heads, n_tokens, head_dim, bf16_out, false, su.n_sms, status,
                            la::kWaitLimitNs, s);
    if (e != cudaSuccess) return cuda_fail(e, "apply launch");
    return la::record_error(LIN_ATTN_OK, "");
}

extern "C" int lin_attn_noalloc_status(struct CUstream_st* stream) {
    DeviceSetup su;
    if (const int rc = device_setup(&su)) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int* status = reinterpret_cast<int*>(su.scratch);
    int word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, status, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the no-alloc status word");
    if (word != 0) {
        e = cudaMemsetAsync(status, 0, sizeof(int), s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the no-alloc status word");
        return la::record_error(LIN_ATTN_ERR_TIMEOUT, "a kernel of an earlier no-alloc call gave up waiting");
    }
    return la::record_error(LIN_ATTN_OK, "");
}
