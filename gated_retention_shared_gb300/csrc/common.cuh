// common.cuh -- element access, gate and launch helpers shared by libyoco's kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "yoco.h"

namespace yoco {

// Lower clamp on log(gamma).  gamma -> 0 (logit -> -inf) would make chunk-local
// cumulative log decays -inf and their differences NaN; e^-30 ~ 1e-13 is zero
// for every tolerance the path is held to.
constexpr float kLogGateMin = -30.0f;

// Workspace status word written by a kernel whose bounded wait gave up:
// kErrMagic | site code.  Anything else means no failure was recorded.
constexpr uint32_t kErrMagic = 0x59434F00u;

typedef uint16_t bf16_t;  // raw bfloat16 bits

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16_t x) { return __uint_as_float(((uint32_t)x) << 16); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16_t from_f32<bf16_t>(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<bf16_t *>(&h);
}

// log(gamma) = logsigmoid(logit) / tau  (paper Section 3.1 Eq. 4; Appendix F takes
// the gate in log space).  logsigmoid(x) = min(x, 0) - log1p(exp(-|x|)).
__device__ __forceinline__ float log_gate(float logit, float inv_tau) {
    float ls = fminf(logit, 0.0f) - log1pf(expf(-fabsf(logit)));
    return fmaxf(ls * inv_tau, kLogGateMin);
}

// Debug builds (-DYOCO_DEBUG_CHECKS, see build.py): kernels check the global indices
// they form from runtime values before they use them.  A failed check records
// kErrMagic | site in this translation unit's debug word (yoco_debug_checks reads
// every unit's word) and the access is skipped: never a trap.  Release builds
// compile every check to `true`.  Sites:
//   0x40 gRet output: a segment's fold reads an E slot    0x41 gRet output: parked-state slot
//   0x42 gRet output: hand-off word                        0x43 gRet segment state: E slot
//   0x44 gRet segment state: G slot                        0x48 append (strip GEMV): cache slot
//   0x49 append (split-K GEMV): cache slot                 0x4A append (CUDA-core GEMM): cache slot
//   0x4B append (tensor-core GEMM): cache slot             0x50 decode attention (tensor cores): key range
//   0x51 decode attention (tensor cores): partial row      0x52 attention (CUDA cores): key range
//   0x53 attention (CUDA cores): output / partial row      0x54 split merge: output row
//   0x58 gRet recurrent step: state element                0x5C GroupNorm + gate: row
//   0x5D rotary encoding: row                              0x5E sliding-window ring: slot
#ifdef YOCO_DEBUG_CHECKS
static __device__ unsigned g_yoco_dbg_word;
__device__ __forceinline__ bool dcheck(bool ok, unsigned site) {
    if (!ok) atomicCAS(&g_yoco_dbg_word, 0u, kErrMagic | site);
    return ok;
}
#define YOCO_DCHECK(cond, site) (::yoco::dcheck((cond), (site)))
#else
#define YOCO_DCHECK(cond, site) (true)
#endif

}  // namespace yoco

// Host accessor of a translation unit's debug word (debug builds only): every .cu
// file with kernels names itself once with YOCO_DEBUG_TU(name).
#ifdef YOCO_DEBUG_CHECKS
#define YOCO_DEBUG_TU(tu)                                                                      \
    namespace yoco_host {                                                                      \
    cudaError_t debug_word_##tu(unsigned *w, int clear) {                                      \
        cudaError_t e = cudaMemcpyFromSymbol(w, ::yoco::g_yoco_dbg_word, sizeof(unsigned));    \
        if (e == cudaSuccess && clear) {                                                       \
            const unsigned zero = 0;                                                           \
            e = cudaMemcpyToSymbol(::yoco::g_yoco_dbg_word, &zero, sizeof(unsigned));          \
        }                                                                                      \
        return e;                                                                              \
    }                                                                                          \
    }
#else
#define YOCO_DEBUG_TU(tu)
#endif

// Host-side status plumbing shared by the API translation units.
namespace yoco_host {
void set_error(const char *fmt, ...);
void count_launches(unsigned n);  // add n to the process-wide launch counter
}  // namespace yoco_host
