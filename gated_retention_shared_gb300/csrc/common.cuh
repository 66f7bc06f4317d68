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

}  // namespace yoco

// Host-side status plumbing shared by the API translation units.
namespace yoco_host {
void set_error(const char *fmt, ...);
void count_launches(unsigned n);  // add n to the process-wide launch counter
}  // namespace yoco_host
