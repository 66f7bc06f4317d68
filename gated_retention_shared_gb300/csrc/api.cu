// api.cu -- the C ABI of libyoco: host-side validation, workspace sizing and
// dispatch to the kernels.  Every check runs before anything is enqueued, so an
// error status means nothing was launched and nothing was written.
#include <atomic>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"

namespace yoco_host {

static thread_local char g_last_error[512] = "";
static std::atomic<uint64_t> g_launches{0};

void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

static std::atomic<int64_t> g_hooks[kHookCount];

int64_t test_hook_value(int hook) {
    return (hook > 0 && hook < kHookCount) ? g_hooks[hook].load(std::memory_order_relaxed) : 0;
}

bool take_injected_failure() {
    int64_t n = g_hooks[kHookFailNextCalls].load(std::memory_order_relaxed);
    while (n > 0)
        if (g_hooks[kHookFailNextCalls].compare_exchange_weak(n, n - 1, std::memory_order_relaxed)) return true;
    return false;
}

int device_sm_count() {
    constexpr int kMaxDev = 64;
    static std::atomic<int> cached[kMaxDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
        (void)cudaGetLastError();
        return kDefaultSmCount;
    }
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return kDefaultSmCount;
    }
    cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

void set_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
}

static yoco_status fail(yoco_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return s;
}

static yoco_status cuda_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) {
        g_last_error[0] = 0;
        return YOCO_OK;
    }
    set_error("%s: %s", what, cudaGetErrorString(e));
    return YOCO_ERR_CUDA;
}

// A pending injected failure (yoco_test_hook) stands in for a failed launch at the
// point where the call would enqueue its first kernel: nothing is launched or written.
#define YOCO_INJECTED_FAILURE(what)                                                     \
    do {                                                                                \
        if (take_injected_failure()) return cuda_status(cudaErrorLaunchFailure, what);  \
    } while (0)

static bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }
static bool valid_dt(yoco_dtype d) { return d == YOCO_F32 || d == YOCO_BF16; }

static yoco_status check_ws(void *ws, size_t have, size_t need) {
    if (need == 0) return YOCO_OK;
    if (!ws) return fail(YOCO_ERR_WORKSPACE, "workspace of %zu bytes required, got NULL", need);
    if (have < need) return fail(YOCO_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", have, need);
    if (!aligned(ws, 256)) return fail(YOCO_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    return YOCO_OK;
}

static yoco_status check_cache(const yoco_kv_cache *c) {
    if (!c) return fail(YOCO_ERR_INVALID_ARG, "cache is NULL");
    if (!c->k || !c->v || !c->len_dev) return fail(YOCO_ERR_INVALID_ARG, "cache k, v and len_dev must be set");
    if (!valid_dt(c->dtype)) return fail(YOCO_ERR_INVALID_ARG, "cache dtype invalid");
    if (c->B <= 0 || c->Hkv <= 0 || c->capacity <= 0)
        return fail(YOCO_ERR_INVALID_ARG, "cache B, Hkv and capacity must be positive");
    if (c->d != 64 && c->d != 128) return fail(YOCO_ERR_UNSUPPORTED, "cache head size %d not in {64, 128}", c->d);
    if (c->len_host < 0 || c->len_host > c->capacity)
        return fail(YOCO_ERR_INVALID_ARG, "cache length %lld outside [0, capacity]", (long long)c->len_host);
    if (!aligned(c->k, 16) || !aligned(c->v, 16)) return fail(YOCO_ERR_INVALID_ARG, "cache k/v must be 16-byte aligned");
    if (c->capacity > (int64_t)INT32_MAX) return fail(YOCO_ERR_UNSUPPORTED, "capacity above 2^31-1");
    if (!(c->rope_base == 0.0f || (c->rope_base > 1.0f && isfinite(c->rope_base))))
        return fail(YOCO_ERR_INVALID_ARG, "rope_base must be 0 (off) or a finite base > 1");
    return YOCO_OK;
}

}  // namespace yoco_host

using namespace yoco_host;

extern "C" {

const char *yoco_status_string(yoco_status s) {
    switch (s) {
    case YOCO_OK: return "ok";
    case YOCO_ERR_INVALID_ARG: return "invalid argument";
    case YOCO_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case YOCO_ERR_CAPACITY: return "cache capacity exceeded";
    case YOCO_ERR_CUDA: return "CUDA error";
    case YOCO_ERR_TIMEOUT: return "on-device wait timed out";
    case YOCO_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    }
    return "unknown status";
}

const char *yoco_last_error(void) { return g_last_error; }

int yoco_version(void) { return YOCO_VERSION; }

yoco_status yoco_workspace_status(void *workspace, int clear, void *stream) {
    if (!workspace) return fail(YOCO_ERR_INVALID_ARG, "workspace is NULL");
    uint32_t word = 0;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_status(e, "workspace_status");
    const bool hit = (word & 0xFFFFFF00u) == yoco::kErrMagic;
    if (clear && hit) {
        e = cudaMemsetAsync(workspace, 0, sizeof(word), st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_status(e, "workspace_status");
    }
    if (hit) return fail(YOCO_ERR_TIMEOUT, "a bounded on-device wait gave up (site %u)", word & 0xFFu);
    g_last_error[0] = 0;
    return YOCO_OK;
}

yoco_status yoco_selftest_wait_timeout(void *workspace, uint64_t limit_ns, void *stream) {
    if (!workspace || !aligned(workspace, 256)) return fail(YOCO_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (limit_ns == 0 || limit_ns > 10000000000ull) return fail(YOCO_ERR_INVALID_ARG, "limit_ns must be in (0, 1e10]");
    return cuda_status(selftest_wait(workspace, limit_ns, (cudaStream_t)stream), "selftest_wait_timeout");
}

yoco_status yoco_selftest_occupy_sms(int ctas, uint64_t ns, void *stream) {
    if (ctas <= 0 || ctas > 4 * device_sm_count()) return fail(YOCO_ERR_INVALID_ARG, "ctas must be in [1, 4 * SMs]");
    if (ns == 0 || ns > 1000000000ull) return fail(YOCO_ERR_INVALID_ARG, "ns must be in (0, 1e9]");
    return cuda_status(selftest_occupy(ctas, ns, (cudaStream_t)stream), "selftest_occupy_sms");
}

uint64_t yoco_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

yoco_status yoco_debug_checks(int clear, uint32_t *word) {
    if (!word) return fail(YOCO_ERR_INVALID_ARG, "word is NULL");
    *word = 0;
#ifdef YOCO_DEBUG_CHECKS
    cudaError_t e = cudaDeviceSynchronize();
    unsigned w = 0;
#define YOCO_READ_DEBUG_WORD(tu)                                   \
    if (e == cudaSuccess) {                                        \
        unsigned x = 0;                                            \
        e = debug_word_##tu(&x, clear);                            \
        if (!w) w = x;                                             \
    }
    YOCO_DEBUG_TUS(YOCO_READ_DEBUG_WORD)
#undef YOCO_READ_DEBUG_WORD
    if (e != cudaSuccess) return cuda_status(e, "debug_checks");
    *word = w;
    g_last_error[0] = 0;
    return YOCO_OK;
#else
    (void)clear;
    return fail(YOCO_ERR_UNSUPPORTED, "libyoco was built without YOCO_DEBUG_CHECKS");
#endif
}

yoco_status yoco_test_hook(int hook, int64_t value) {
    if (hook == YOCO_HOOK_FAIL_NEXT_CALLS) {
        if (value < 0 || value > 1000000) return fail(YOCO_ERR_INVALID_ARG, "failure count must be in [0, 1e6]");
    } else if (hook == YOCO_HOOK_GRET_SEG0_DELAY_NS) {
        if (value < 0 || value > 1000000000) return fail(YOCO_ERR_INVALID_ARG, "delay must be in [0, 1e9] ns");
    } else if (hook == YOCO_HOOK_GRET_SEGMENTS) {
        if (value < 0 || value > 4096) return fail(YOCO_ERR_INVALID_ARG, "segment count must be in [0, 4096]");
    } else {
        return fail(YOCO_ERR_INVALID_ARG, "unknown test hook %d", hook);
    }
    g_hooks[hook].store(value, std::memory_order_relaxed);
    g_last_error[0] = 0;
    return YOCO_OK;
}

// ----------------------------------------------------------------------- gRet

static yoco_status check_gret_shapes(int B, int N, int H, int dk, int dv, yoco_dtype in_dt, yoco_dtype out_dt) {
    if (B <= 0 || H <= 0 || N < 0) return fail(YOCO_ERR_INVALID_ARG, "B, H must be > 0 and N >= 0");
    if (!valid_dt(in_dt) || !valid_dt(out_dt)) return fail(YOCO_ERR_INVALID_ARG, "dtype invalid");
    if (in_dt != out_dt) return fail(YOCO_ERR_UNSUPPORTED, "in_dt must equal out_dt");
    if (dk != dv || (dk != 64 && dk != 128)) return fail(YOCO_ERR_UNSUPPORTED, "need dk == dv in {64, 128}");
    if ((int64_t)B * N * H * dk > ((int64_t)1 << 40)) return fail(YOCO_ERR_UNSUPPORTED, "tensor too large");
    return YOCO_OK;
}

size_t yoco_gret_prefill_workspace_size(int B, int N, int H, int dk, int dv, int chunk, yoco_dtype in_dt) {
    if (check_gret_shapes(B, N, H, dk, dv, in_dt, in_dt) != YOCO_OK || N == 0) return 0;
    bool tc = (chunk == 0 || chunk == 128) && gret_tc_eligible(B, N, H, dk, dv, in_dt);
    return tc ? gret_tc_workspace(B, N, H, dk, dv) : gret_simt_workspace(B, N, H, dk, dv);
}

yoco_status yoco_gret_prefill_chunkwise(const void *q, const void *k, const void *v, const float *gate_logits,
                                        float tau, void *o, float *state, int B, int N, int H, int dk, int dv,
                                        int chunk, yoco_dtype in_dt, yoco_dtype out_dt, void *workspace,
                                        size_t ws_bytes, void *stream) {
    yoco_status s = check_gret_shapes(B, N, H, dk, dv, in_dt, out_dt);
    if (s != YOCO_OK) return s;
    if (!state) return fail(YOCO_ERR_INVALID_ARG, "state is NULL");
    if (!(tau > 0.0f) || !isfinite(tau)) return fail(YOCO_ERR_INVALID_ARG, "tau must be finite and > 0");
    if (chunk != 0 && chunk != 64 && chunk != 128)
        return fail(YOCO_ERR_UNSUPPORTED, "chunk %d not in {0, 64, 128}", chunk);
    if (N == 0) return YOCO_OK;
    if (!q || !k || !v || !gate_logits || !o) return fail(YOCO_ERR_INVALID_ARG, "null tensor");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(state, 16))
        return fail(YOCO_ERR_INVALID_ARG, "q, k, v, o, state must be 16-byte aligned");
    const bool tc = (chunk == 0 || chunk == 128) && gret_tc_eligible(B, N, H, dk, dv, in_dt);
    const size_t need = tc ? gret_tc_workspace(B, N, H, dk, dv) : gret_simt_workspace(B, N, H, dk, dv);
    if ((s = check_ws(workspace, ws_bytes, need)) != YOCO_OK) return s;
    YOCO_INJECTED_FAILURE("gret_prefill_chunkwise");
    GretArgs a{q, k, v, gate_logits, tau, o, state, B, N, H, dk, dv, in_dt};
    cudaStream_t st = (cudaStream_t)stream;
    return cuda_status(tc ? gret_prefill_tc(a, nullptr, workspace, st) : gret_prefill_simt(a, workspace, st),
                       "gret_prefill_chunkwise");
}

yoco_status yoco_gret_prefill_chunkwise_gn_gate(const void *q, const void *k, const void *v, const float *gate_logits,
                                                float tau, const void *gate, const float *gn_weight,
                                                const float *gn_bias, float eps, void *z, float *state, int B, int N,
                                                int H, int dk, int dv, yoco_dtype dt, void *workspace,
                                                size_t ws_bytes, void *stream) {
    yoco_status s = check_gret_shapes(B, N, H, dk, dv, dt, dt);
    if (s != YOCO_OK) return s;
    if (!state) return fail(YOCO_ERR_INVALID_ARG, "state is NULL");
    if (!(tau > 0.0f) || !isfinite(tau)) return fail(YOCO_ERR_INVALID_ARG, "tau must be finite and > 0");
    if (!(eps > 0.f) || !isfinite(eps)) return fail(YOCO_ERR_INVALID_ARG, "eps must be finite and > 0");
    if (N == 0) return YOCO_OK;
    if (!q || !k || !v || !gate_logits || !gate || !z) return fail(YOCO_ERR_INVALID_ARG, "null tensor");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(z, 16) || !aligned(gate, 16) ||
        !aligned(state, 16))
        return fail(YOCO_ERR_INVALID_ARG, "q, k, v, gate, z, state must be 16-byte aligned");
    const bool tc = gret_tc_eligible(B, N, H, dk, dv, dt);
    const size_t need = tc ? gret_tc_workspace(B, N, H, dk, dv) : gret_simt_workspace(B, N, H, dk, dv);
    if ((s = check_ws(workspace, ws_bytes, need)) != YOCO_OK) return s;
    YOCO_INJECTED_FAILURE("gret_prefill_chunkwise_gn_gate");
    GretArgs a{q, k, v, gate_logits, tau, z, state, B, N, H, dk, dv, dt};
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e;
    if (tc) {
        const GnArgs gn{gate, gn_weight, gn_bias, eps};
        e = gret_prefill_tc(a, &gn, workspace, st);
    } else {
        // the CUDA-core kernel writes the retention output into z, then Eq. 7 in place
        e = gret_prefill_simt(a, workspace, st);
        if (e == cudaSuccess) e = group_norm_gate(z, gate, gn_weight, gn_bias, eps, z, (int64_t)B * N * H, H, dv, dt, st);
    }
    return cuda_status(e, "gret_prefill_chunkwise_gn_gate");
}

yoco_status yoco_gret_decode_step(const void *q, const void *k, const void *v, const float *gate_logits, float tau,
                                  float *state, void *o, int B, int H, int dk, int dv, yoco_dtype in_dt,
                                  yoco_dtype out_dt, void *stream) {
    yoco_status s = check_gret_shapes(B, 1, H, dk, dv, in_dt, out_dt);
    if (s != YOCO_OK) return s;
    if (!q || !k || !v || !gate_logits || !state || !o) return fail(YOCO_ERR_INVALID_ARG, "null tensor");
    if (!(tau > 0.0f) || !isfinite(tau)) return fail(YOCO_ERR_INVALID_ARG, "tau must be finite and > 0");
    if (!aligned(state, 16)) return fail(YOCO_ERR_INVALID_ARG, "state must be 16-byte aligned");
    YOCO_INJECTED_FAILURE("gret_decode_step");
    return cuda_status(gret_decode(q, k, v, gate_logits, tau, state, o, B, H, dk, dv, in_dt, (cudaStream_t)stream),
                       "gret_decode_step");
}

// ------------------------------------------------------------------ shared KV

size_t yoco_shared_kv_workspace_size(int B, int T, int dm, const yoco_kv_cache *cache) {
    if (!cache || B <= 0 || T <= 0 || dm <= 0) return 0;
    return kv_proj_workspace(B, T, dm, cache->Hkv, cache->d, cache->dtype, cache->rope_base);
}

yoco_status yoco_shared_kv_project_append(const void *M, const void *rms_w, float eps, const void *Wk,
                                          const void *Wv, int T, int dm, yoco_kv_cache *cache, void *workspace,
                                          size_t ws_bytes, void *stream) {
    yoco_status s = check_cache(cache);
    if (s != YOCO_OK) return s;
    if (T <= 0 || dm <= 0) return fail(YOCO_ERR_INVALID_ARG, "T and dm must be > 0");
    if (!M || !Wk || !Wv) return fail(YOCO_ERR_INVALID_ARG, "null tensor");
    if (!(eps >= 0.0f) || !isfinite(eps)) return fail(YOCO_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (!aligned(M, 16) || !aligned(Wk, 16) || !aligned(Wv, 16) || (rms_w && !aligned(rms_w, 16)))
        return fail(YOCO_ERR_INVALID_ARG, "M, Wk, Wv and rms_w must be 16-byte aligned");
    if (cache->len_host + T > cache->capacity)
        return fail(YOCO_ERR_CAPACITY, "append of %d tokens at length %lld exceeds capacity %lld", T,
                    (long long)cache->len_host, (long long)cache->capacity);
    if ((int64_t)cache->B * T > INT32_MAX) return fail(YOCO_ERR_UNSUPPORTED, "B*T too large");
    const size_t need = kv_proj_workspace(cache->B, T, dm, cache->Hkv, cache->d, cache->dtype, cache->rope_base);
    if ((s = check_ws(workspace, ws_bytes, need)) != YOCO_OK) return s;
    YOCO_INJECTED_FAILURE("shared_kv_project_append");
    KvProjArgs a{M, rms_w, Wk, Wv, eps, cache->B, T, dm, cache->Hkv, cache->d, cache->capacity, cache->len_host,
                 cache->k, cache->v, cache->len_dev, cache->dtype, cache->rope_base};
    s = cuda_status(kv_project_append(a, workspace, (cudaStream_t)stream), "shared_kv_project_append");
    if (s == YOCO_OK) cache->len_host += T;
    return s;
}

// ------------------------------------------------------------ cross attention

size_t yoco_cross_attn_workspace_size(int B, int Hq, int T, const yoco_kv_cache *cache, int num_splits) {
    if (!cache || B <= 0 || Hq <= 0 || T <= 0 || cache->Hkv <= 0) return 0;
    int splits = num_splits > 0 ? num_splits
                                : attn_auto_splits(B, cache->Hkv, cache->capacity,
                                                   attn_ctas_per_sm(cache->dtype, cache->d, Hq / cache->Hkv));
    if (T > 1 && num_splits <= 0) splits = 1;
    return attn_workspace(B, Hq, T, cache->d, splits);
}

static yoco_status attn_common(const void *Q, int Hq, int T, int64_t p0, const yoco_kv_cache *cache, float scale,
                               int num_splits, void *O, void *ws, size_t ws_bytes, void *stream) {
    yoco_status s = check_cache(cache);
    if (s != YOCO_OK) return s;
    if (!Q || !O) return fail(YOCO_ERR_INVALID_ARG, "null tensor");
    if (Hq <= 0 || Hq % cache->Hkv != 0) return fail(YOCO_ERR_UNSUPPORTED, "Hq must be a positive multiple of Hkv");
    if (Hq / cache->Hkv > 16) return fail(YOCO_ERR_UNSUPPORTED, "at most 16 query heads per kv head");
    if (T <= 0) return fail(YOCO_ERR_INVALID_ARG, "T must be > 0");
    if (p0 < 0 || p0 + T > cache->len_host)
        return fail(YOCO_ERR_INVALID_ARG, "rows at positions [%lld, %lld) are not all in the cache (length %lld)",
                    (long long)p0, (long long)(p0 + T), (long long)cache->len_host);
    if (!isfinite(scale)) return fail(YOCO_ERR_INVALID_ARG, "scale must be finite");
    if (!aligned(Q, 16) || !aligned(O, 16)) return fail(YOCO_ERR_INVALID_ARG, "Q/O must be 16-byte aligned");
    if (num_splits < 0) return fail(YOCO_ERR_INVALID_ARG, "num_splits must be >= 0");
    const int64_t keys = p0 + T;
    int splits = num_splits > 0 ? num_splits
                                : (T == 1 ? attn_auto_splits(cache->B, cache->Hkv, keys,
                                                             attn_ctas_per_sm(cache->dtype, cache->d, Hq / cache->Hkv))
                                          : 1);
    if (splits > 4096) return fail(YOCO_ERR_UNSUPPORTED, "num_splits above 4096");
    const size_t need = attn_workspace(cache->B, Hq, T, cache->d, splits);
    if ((s = check_ws(ws, ws_bytes, need)) != YOCO_OK) return s;
    YOCO_INJECTED_FAILURE("cross_attn");
    AttnArgs a{Q, O, cache->k, cache->v, cache->B, T, Hq, cache->Hkv, cache->d, cache->capacity, p0, scale,
               cache->dtype, cache->rope_base};
    return cuda_status(attn_run(a, splits, ws, (cudaStream_t)stream), "cross_attn");
}

yoco_status yoco_cross_attn_prefill(const void *Q, int Hq, int T, int64_t p0, const yoco_kv_cache *cache, float scale,
                                    void *O, void *workspace, size_t ws_bytes, void *stream) {
    return attn_common(Q, Hq, T, p0, cache, scale, T == 1 ? 0 : 1, O, workspace, ws_bytes, stream);
}

yoco_status yoco_cross_attn_decode(const void *Q, int Hq, const yoco_kv_cache *cache, float scale, int num_splits,
                                   void *O, void *workspace, size_t ws_bytes, void *stream) {
    yoco_status s = check_cache(cache);
    if (s != YOCO_OK) return s;
    if (cache->len_host < 1) return fail(YOCO_ERR_INVALID_ARG, "decode needs a non-empty cache");
    return attn_common(Q, Hq, 1, cache->len_host - 1, cache, scale, num_splits, O, workspace, ws_bytes, stream);
}

// ---------------------------------------------- gated retention output (Eq. 7)

yoco_status yoco_gret_decode_step_gn_gate(const void *q, const void *k, const void *v, const float *gate_logits,
                                          float tau, float *state, const void *gate, const float *gn_weight,
                                          const float *gn_bias, float eps, void *z, int B, int H, int dk, int dv,
                                          yoco_dtype dt, void *stream) {
    yoco_status s = check_gret_shapes(B, 1, H, dk, dv, dt, dt);
    if (s != YOCO_OK) return s;
    if (!q || !k || !v || !gate_logits || !state || !gate || !z) return fail(YOCO_ERR_INVALID_ARG, "null tensor");
    if (dv != 64 && dv != 128) return fail(YOCO_ERR_UNSUPPORTED, "dv %d not in {64, 128}", dv);
    if (!(tau > 0.0f) || !isfinite(tau)) return fail(YOCO_ERR_INVALID_ARG, "tau must be finite and > 0");
    if (!(eps > 0.f) || !isfinite(eps)) return fail(YOCO_ERR_INVALID_ARG, "eps must be finite and > 0");
    if (!aligned(state, 16)) return fail(YOCO_ERR_INVALID_ARG, "state must be 16-byte aligned");
    YOCO_INJECTED_FAILURE("gret_decode_step_gn_gate");
    return cuda_status(gret_decode_gn(q, k, v, gate_logits, tau, state, gate, gn_weight, gn_bias, eps, z, B, H, dk, dv,
                                      dt, (cudaStream_t)stream),
                       "gret_decode_step_gn_gate");
}

yoco_status yoco_gret_group_norm_gate(const void *o, const void *gate, const float *gn_weight, const float *gn_bias,
                                      float eps, void *z, int B, int N, int H, int d, yoco_dtype dt, void *stream) {
    if (!o || !gate || !z) return fail(YOCO_ERR_INVALID_ARG, "null tensor");
    if (!valid_dt(dt)) return fail(YOCO_ERR_INVALID_ARG, "dtype invalid");
    if (d != 64 && d != 128) return fail(YOCO_ERR_UNSUPPORTED, "head size %d not in {64, 128}", d);
    if (B <= 0 || N < 0 || H <= 0) return fail(YOCO_ERR_INVALID_ARG, "B, H must be > 0 and N >= 0");
    if (!(eps > 0.f) || !isfinite(eps)) return fail(YOCO_ERR_INVALID_ARG, "eps must be finite and > 0");
    if (!aligned(o, 16) || !aligned(gate, 16) || !aligned(z, 16))
        return fail(YOCO_ERR_INVALID_ARG, "o, gate, z must be 16-byte aligned");
    YOCO_INJECTED_FAILURE("gret_group_norm_gate");
    return cuda_status(group_norm_gate(o, gate, gn_weight, gn_bias, eps, z, (int64_t)B * N * H, H, d, dt,
                                       (cudaStream_t)stream),
                       "gret_group_norm_gate");
}

// ------------------------------------ gated-retention input projections (one GEMM)

size_t yoco_gret_qkvg_workspace_size(int B, int N, int H, int d, float rope_base) {
    (void)B; (void)H;
    if (N <= 0 || d <= 0) return 256;
    return 256 + (rope_base > 0.f ? (size_t)N * (d / 2) * sizeof(float2) : 0);
}

yoco_status yoco_gret_qkvg_project(const void *X, const void *W, int B, int N, int dm, int H, int d, int64_t pos0,
                                   float rope_base, void *q, void *k, void *v, float *gate_logits, void *workspace,
                                   size_t ws_bytes, void *stream) {
    if (!X || !W || !q || !k || !v || !gate_logits) return fail(YOCO_ERR_INVALID_ARG, "null tensor");
    if (B <= 0 || N < 0 || dm <= 0 || H <= 0) return fail(YOCO_ERR_INVALID_ARG, "B, dm, H must be > 0 and N >= 0");
    if (d != 64 && d != 128) return fail(YOCO_ERR_UNSUPPORTED, "head size %d not in {64, 128}", d);
    if (dm % 8 != 0 || H % 8 != 0)
        return fail(YOCO_ERR_UNSUPPORTED, "dm and H must be multiples of 8 (16-byte rows of X and W)");
    if ((int64_t)B * N > INT32_MAX / 2 || (int64_t)H * d * 3 + H > INT32_MAX / 2)
        return fail(YOCO_ERR_UNSUPPORTED, "size out of range");
    if (pos0 < 0) return fail(YOCO_ERR_INVALID_ARG, "pos0 must be >= 0");
    if (!(rope_base == 0.0f || (rope_base > 1.0f && isfinite(rope_base))))
        return fail(YOCO_ERR_INVALID_ARG, "rope_base must be 0 (off) or a finite base > 1");
    if (!aligned(X, 16) || !aligned(W, 16) || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16))
        return fail(YOCO_ERR_INVALID_ARG, "X, W, q, k, v must be 16-byte aligned");
    yoco_status s = check_ws(workspace, ws_bytes, yoco_gret_qkvg_workspace_size(B, N, H, d, rope_base));
    if (s != YOCO_OK) return s;
    if (N == 0) return YOCO_OK;
    YOCO_INJECTED_FAILURE("gret_qkvg_project");
    cudaStream_t st = (cudaStream_t)stream;
    float2 *rope_cs = nullptr;
    cudaError_t e = cudaSuccess;
    if (rope_base > 0.f) {
        rope_cs = reinterpret_cast<float2 *>((char *)workspace + 256);
        e = rope_table(rope_cs, pos0, N, d, rope_base, st);
    }
    if (e == cudaSuccess) e = qkvg_project(X, W, B, N, dm, H, d, q, k, v, gate_logits, rope_cs, (int *)workspace, st);
    return cuda_status(e, "gret_qkvg_project");
}

// -------------------------------------------------- rotary position encoding

yoco_status yoco_rope_apply(void *x, int B, int N, int H, int d, int64_t pos0, float base, yoco_dtype dt,
                            void *stream) {
    if (!x) return fail(YOCO_ERR_INVALID_ARG, "null tensor");
    if (!valid_dt(dt)) return fail(YOCO_ERR_INVALID_ARG, "dtype invalid");
    if (d != 64 && d != 128) return fail(YOCO_ERR_UNSUPPORTED, "head size %d not in {64, 128}", d);
    if (B <= 0 || N < 0 || H <= 0 || B > 65535) return fail(YOCO_ERR_INVALID_ARG, "B in [1, 65535], H > 0, N >= 0");
    if (pos0 < 0) return fail(YOCO_ERR_INVALID_ARG, "pos0 must be >= 0");
    if (!(base > 1.0f) || !isfinite(base)) return fail(YOCO_ERR_INVALID_ARG, "base must be finite and > 1");
    if (!aligned(x, 16)) return fail(YOCO_ERR_INVALID_ARG, "x must be 16-byte aligned");
    YOCO_INJECTED_FAILURE("rope_apply");
    return cuda_status(rope_apply(x, B, N, H, d, pos0, base, dt, (cudaStream_t)stream), "rope_apply");
}

// ------------------------------------------------ sliding-window self-decoder

static yoco_status check_ring(const yoco_swa_ring *r, int Hq) {
    if (!r) return fail(YOCO_ERR_INVALID_ARG, "ring is NULL");
    if (!r->k || !r->v) return fail(YOCO_ERR_INVALID_ARG, "ring k and v must be set");
    if (!valid_dt(r->dtype)) return fail(YOCO_ERR_INVALID_ARG, "ring dtype invalid");
    if (r->B <= 0 || r->Hkv <= 0 || r->window <= 0) return fail(YOCO_ERR_INVALID_ARG, "ring B, Hkv and window must be positive");
    if (r->d != 64 && r->d != 128) return fail(YOCO_ERR_UNSUPPORTED, "ring head size %d not in {64, 128}", r->d);
    if (r->pos < 0) return fail(YOCO_ERR_INVALID_ARG, "ring position must be >= 0");
    if (!aligned(r->k, 16) || !aligned(r->v, 16)) return fail(YOCO_ERR_INVALID_ARG, "ring k/v must be 16-byte aligned");
    if (Hq <= 0 || Hq % r->Hkv != 0) return fail(YOCO_ERR_UNSUPPORTED, "Hq must be a positive multiple of Hkv");
    if (Hq / r->Hkv > 16) return fail(YOCO_ERR_UNSUPPORTED, "at most 16 query heads per kv head");
    return YOCO_OK;
}

size_t yoco_swa_workspace_size(int B, int Hq, const yoco_swa_ring *ring) {
    if (!ring || B <= 0 || Hq <= 0 || ring->Hkv <= 0 || ring->window <= 0) return 0;
    const int splits = attn_auto_splits(B, ring->Hkv, ring->window, attn_ctas_per_sm(ring->dtype, ring->d, Hq / ring->Hkv));
    return attn_workspace(B, Hq, 1, ring->d, splits);
}

yoco_status yoco_swa_prefill(const void *q, const void *k, const void *v, int Hq, int N, float scale, void *o,
                             yoco_swa_ring *ring, void *workspace, size_t ws_bytes, void *stream) {
    yoco_status s = check_ring(ring, Hq);
    if (s != YOCO_OK) return s;
    if (!q || !k || !v || !o) return fail(YOCO_ERR_INVALID_ARG, "null tensor");
    if (N < 0) return fail(YOCO_ERR_INVALID_ARG, "N must be >= 0");
    if (ring->pos != 0) return fail(YOCO_ERR_INVALID_ARG, "prefill starts a sequence: ring position must be 0");
    if (ring->dtype != YOCO_BF16 || ring->d != 128)
        return fail(YOCO_ERR_UNSUPPORTED, "sliding-window prefill runs in bf16 with head size 128");
    if (!isfinite(scale)) return fail(YOCO_ERR_INVALID_ARG, "scale must be finite");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
        return fail(YOCO_ERR_INVALID_ARG, "q, k, v, o must be 16-byte aligned");
    if ((int64_t)ring->B * Hq > 0x7fffffff || N > (1 << 30)) return fail(YOCO_ERR_UNSUPPORTED, "size out of range");
    if ((s = check_ws(workspace, ws_bytes, 256)) != YOCO_OK) return s;
    if (N == 0) return YOCO_OK;
    YOCO_INJECTED_FAILURE("swa_prefill");
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = swa_fa_launch(q, k, v, o, ring->B, N, Hq, ring->Hkv, ring->window, scale, (int *)workspace, st);
    if (e == cudaSuccess) {
        // the ring keeps the last `window` tokens for decoding
        const int n = N < ring->window ? N : ring->window;
        e = swa_ring_write(k, v, ring->k, ring->v, ring->B, N, ring->Hkv, ring->d, ring->window, N - n, n, N - n,
                           ring->dtype, st);
    }
    if (e != cudaSuccess) return cuda_status(e, "swa_prefill");
    ring->pos = N;
    return YOCO_OK;
}

yoco_status yoco_swa_decode(const void *q, const void *k, const void *v, int Hq, float scale, void *o,
                            yoco_swa_ring *ring, void *workspace, size_t ws_bytes, void *stream) {
    yoco_status s = check_ring(ring, Hq);
    if (s != YOCO_OK) return s;
    if (!q || !k || !v || !o) return fail(YOCO_ERR_INVALID_ARG, "null tensor");
    if (!isfinite(scale)) return fail(YOCO_ERR_INVALID_ARG, "scale must be finite");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
        return fail(YOCO_ERR_INVALID_ARG, "q, k, v, o must be 16-byte aligned");
    // keys in the ring after this token: positions max(0, pos - window + 1) .. pos
    const int64_t keys = ring->pos + 1 < ring->window ? ring->pos + 1 : ring->window;
    const int splits =
        attn_auto_splits(ring->B, ring->Hkv, keys, attn_ctas_per_sm(ring->dtype, ring->d, Hq / ring->Hkv));
    if ((s = check_ws(workspace, ws_bytes, attn_workspace(ring->B, Hq, 1, ring->d, splits))) != YOCO_OK) return s;
    YOCO_INJECTED_FAILURE("swa_decode");
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = swa_ring_write(k, v, ring->k, ring->v, ring->B, 1, ring->Hkv, ring->d, ring->window, 0, 1,
                                   ring->pos, ring->dtype, st);
    if (e == cudaSuccess) {
        // the filled slots, in whatever order the ring holds them: every one is in the window
        AttnArgs a{q, o, ring->k, ring->v, ring->B, 1, Hq, ring->Hkv, ring->d, ring->window, keys - 1, scale,
                   ring->dtype, 0.0f};
        e = attn_run(a, splits, workspace, st);
    }
    if (e != cudaSuccess) return cuda_status(e, "swa_decode");
    ring->pos += 1;
    return YOCO_OK;
}

}  // extern "C"
