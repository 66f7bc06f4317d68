// gn_gate.cu -- output of multi-head gated retention (paper Section 3.1, Eq. 7):
//     Y = GroupNorm_h(Concat(head_1..head_H)),   z = swish(X W_G) (.) Y
// One group per head: a token's head vector is centred and scaled by
// 1 / sqrt(variance + eps) (variance over the head's d channels), then w, b per
// channel.  The gate's pre-activation X W_G comes from the caller.
//
// One warp per (token, head) row: lane l holds channels l * V .. l * V + V - 1
// (V = d / 32), the mean and the variance (of the centred values) are warp
// reductions, so every row is read once and written once: HBM-bound at
// 3 * d * elem bytes per row.  z may be o (each warp reads its row before writing).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace yoco {

// V consecutive elements (V * sizeof(T) = 4, 8 or 16 bytes, aligned) as one access
template <typename T, int V>
__device__ __forceinline__ void load_v(const T *p, float (&x)[V]) {
    if constexpr (sizeof(T) == 2 && V == 4) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xFFFF0000u);
        x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xFFFF0000u);
    } else if constexpr (sizeof(T) == 2 && V == 2) {
        const uint32_t u = *reinterpret_cast<const uint32_t *>(p);
        x[0] = __uint_as_float(u << 16); x[1] = __uint_as_float(u & 0xFFFF0000u);
    } else if constexpr (V == 4) {
        const float4 f = *reinterpret_cast<const float4 *>(p);
        x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
    } else {
        const float2 f = *reinterpret_cast<const float2 *>(p);
        x[0] = f.x; x[1] = f.y;
    }
}

template <typename T, int V>
__device__ __forceinline__ void store_v(T *p, const float (&y)[V]) {
    if constexpr (sizeof(T) == 2) {
        uint32_t u[V / 2];
#pragma unroll
        for (int i = 0; i < V / 2; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(y[2 * i], y[2 * i + 1]);
            u[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        if constexpr (V == 4) *reinterpret_cast<uint2 *>(p) = make_uint2(u[0], u[1]);
        else *reinterpret_cast<uint32_t *>(p) = u[0];
    } else if constexpr (V == 4) {
        *reinterpret_cast<float4 *>(p) = make_float4(y[0], y[1], y[2], y[3]);
    } else {
        *reinterpret_cast<float2 *>(p) = make_float2(y[0], y[1]);
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(256)
group_norm_gate_kernel(const T *o, const T *__restrict__ gate, const float *__restrict__ w,
                       const float *__restrict__ bias, float eps, T *z, int64_t rows, int H) {
    constexpr int V = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t row = blockIdx.x * (int64_t)(blockDim.x / 32) + threadIdx.x / 32; row < rows; row += warps) {
        if (!YOCO_DCHECK(row < rows, 0x5C)) break;
        const size_t base = (size_t)row * D + (size_t)lane * V;
        float x[V], g[V];
        load_v<T, V>(o + base, x);
        load_v<T, V>(gate + base, g);
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < V; ++i) s += x[i];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        const float mean = s * (1.f / D);
        float q = 0.f;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            x[i] -= mean;
            q = fmaf(x[i], x[i], q);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) q += __shfl_xor_sync(0xffffffffu, q, off);
        const float inv = rsqrtf(q * (1.f / D) + eps);
        const int h = (int)(row % H);
        float out[V];
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int c = lane * V + i;
            float y = x[i] * inv;
            if (w) y *= w[(size_t)h * D + c];
            if (bias) y += bias[(size_t)h * D + c];
            const float sw = g[i] / (1.f + __expf(-g[i]));  // swish(g) = g sigmoid(g)
            out[i] = sw * y;
        }
        store_v<T, V>(z + base, out);
    }
}

}  // namespace yoco

namespace yoco_host {
using namespace yoco;

cudaError_t group_norm_gate(const void *o, const void *gate, const float *w, const float *b, float eps, void *z,
                            int64_t rows, int H, int d, yoco_dtype dt, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    const int blocks = (int)std::min<int64_t>((rows + 7) / 8, (int64_t)device_sm_count() * 16);
    count_launches(1);
#define YOCO_GN(T_, D_)                                                                                             \
    group_norm_gate_kernel<T_, D_><<<blocks, 256, 0, st>>>((const T_ *)o, (const T_ *)gate, w, b, eps, (T_ *)z,    \
                                                           rows, H)
    if (dt == YOCO_BF16) {
        if (d == 128) YOCO_GN(bf16_t, 128);
        else YOCO_GN(bf16_t, 64);
    } else {
        if (d == 128) YOCO_GN(float, 128);
        else YOCO_GN(float, 64);
    }
#undef YOCO_GN
    return cudaGetLastError();
}

}  // namespace yoco_host

YOCO_DEBUG_TU(gn_gate)
