// attn_noalloc.cu -- split-KV cross-attention decode for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they decode: a host runtime that forbids allocation after start-up, a
// real-time serving loop whose memory budget is fixed in advance, a plugin that
// is handed only its input and output buffers.  yoco_cross_attn_decode needs a
// caller-provided workspace for its per-split partial results; this variant
// keeps that scratch in a fixed-size array that lives in the library's device
// image instead, so the caller passes only Q, the cache and O.
//
// The array (kNoAllocScratchBytes) is created by the CUDA runtime on every GPU
// that loads libyoco and stays there until the process exits.  All calls on a
// device share it and it keeps whatever the previous call wrote; this kernel
// writes every partial it later reads, so nothing has to be cleared.  Two calls
// that run at the same time on one device (different streams) race on it.
#include <stdio.h>

#include "common.cuh"
#include "kernels.h"

namespace yoco_host {
void set_error(const char *fmt, ...);
}

namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB = 1,048,576 fp32 partials
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device.  In host code
// `g_noalloc_scratch` is only a host-side stand-in; the kernel must be given the
// address the runtime reports.  Looked up on every call (no allocation, no stream
// work), so a context that was torn down and re-created gets its own address.  The
// first lookup on a device may load the library's device code there, which is why
// that first call should come before any stream capture on the device.
cudaError_t scratch_for_current_device(void **out) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    *out = p;
    return cudaSuccess;
}

yoco_status reject(yoco_status s, const char *msg, long long a = 0, long long b = 0) {
    yoco_host::set_error(msg, a, b);
    return s;
}

}  // namespace

extern "C" YOCO_API yoco_status yoco_cross_attn_decode_noalloc(const void *Q, int Hq, const yoco_kv_cache *cache,
                                                              float scale, int num_splits, void *O, void *stream) {
    using namespace yoco_host;
    if (!cache || !cache->k || !cache->v || !cache->len_dev || !Q || !O)
        return reject(YOCO_ERR_INVALID_ARG, "null tensor or cache");
    if (cache->dtype != YOCO_F32 && cache->dtype != YOCO_BF16) return reject(YOCO_ERR_INVALID_ARG, "cache dtype invalid");
    if (cache->B <= 0 || cache->Hkv <= 0 || cache->capacity <= 0 || cache->capacity > (int64_t)INT32_MAX)
        return reject(YOCO_ERR_INVALID_ARG, "cache B, Hkv or capacity out of range");
    if (cache->d != 64 && cache->d != 128) return reject(YOCO_ERR_UNSUPPORTED, "cache head size %lld not in {64, 128}", cache->d);
    if (!(cache->rope_base == 0.0f || (cache->rope_base > 1.0f && isfinite(cache->rope_base))))
        return reject(YOCO_ERR_INVALID_ARG, "rope_base must be 0 (off) or a finite base > 1");
    if (cache->len_host < 1 || cache->len_host > cache->capacity)
        return reject(YOCO_ERR_INVALID_ARG, "decode needs 1 <= length (%lld) <= capacity", cache->len_host);
    if (Hq <= 0 || Hq % cache->Hkv != 0 || Hq / cache->Hkv > 16)
        return reject(YOCO_ERR_UNSUPPORTED, "Hq must be a multiple of Hkv with at most 16 query heads per kv head");
    if (((uintptr_t)Q | (uintptr_t)O | (uintptr_t)cache->k | (uintptr_t)cache->v) % 16 != 0)
        return reject(YOCO_ERR_INVALID_ARG, "Q, O and cache k/v must be 16-byte aligned");
    if (!isfinite(scale)) return reject(YOCO_ERR_INVALID_ARG, "scale must be finite");
    if (num_splits < 0) return reject(YOCO_ERR_INVALID_ARG, "num_splits must be >= 0");
    if (num_splits > 4096) return reject(YOCO_ERR_UNSUPPORTED, "num_splits above 4096");

    const int64_t keys = cache->len_host;
    int splits = num_splits;
    if (splits == 0) {
        // automatic: the usual split count, reduced until the partials fit the scratch
        splits = attn_auto_splits(cache->B, cache->Hkv, keys, attn_ctas_per_sm(cache->dtype, cache->d, Hq / cache->Hkv));
        while (splits > 1 && attn_workspace(cache->B, Hq, 1, cache->d, splits) > kNoAllocScratchBytes) --splits;
    }
    const size_t need = attn_workspace(cache->B, Hq, 1, cache->d, splits);
    if (need > kNoAllocScratchBytes)
        return reject(YOCO_ERR_UNSUPPORTED,
                      "num_splits needs %lld bytes of scratch; the built-in scratch holds %lld bytes "
                      "(use fewer splits or yoco_cross_attn_decode with a workspace)",
                      (long long)need, (long long)kNoAllocScratchBytes);

    if (take_injected_failure()) {
        set_error("cross_attn_decode_noalloc: %s", cudaGetErrorString(cudaErrorLaunchFailure));
        return YOCO_ERR_CUDA;
    }
    void *scratch = nullptr;
    cudaError_t e = scratch_for_current_device(&scratch);
    if (e != cudaSuccess) {
        set_error("cross_attn_decode_noalloc: scratch lookup failed: %s", cudaGetErrorString(e));
        return YOCO_ERR_CUDA;
    }
    AttnArgs a{Q, O, cache->k, cache->v, cache->B, 1, Hq, cache->Hkv, cache->d, cache->capacity, keys - 1, scale,
               cache->dtype, cache->rope_base};
    e = attn_run(a, splits, scratch, (cudaStream_t)stream);
    if (e != cudaSuccess) {
        set_error("cross_attn_decode_noalloc: %s", cudaGetErrorString(e));
        return YOCO_ERR_CUDA;
    }
    return YOCO_OK;
}

extern "C" YOCO_API yoco_status yoco_cross_attn_decode_noalloc_status(int clear, void *stream) {
    using namespace yoco_host;
    void *scratch = nullptr;
    cudaError_t e = scratch_for_current_device(&scratch);
    if (e != cudaSuccess) {
        set_error("cross_attn_decode_noalloc_status: scratch lookup failed: %s", cudaGetErrorString(e));
        return YOCO_ERR_CUDA;
    }
    // the status word sits where a workspace keeps it: the scratch's first bytes
    return yoco_workspace_status(scratch, clear, stream);
}
