// rope.cu -- rotary position encoding of token-major q or k in place (paper
// Section 3.1: Q (.) Theta, K (.) conj(Theta); the gRet and sliding-window
// self-decoders rotate their own q and k before their token mixer).  Channel pair
// (2i, 2i+1) of row n (every head, every sequence) turns by (pos0 + n) theta_i.
//
// One CTA per 128 rows of one sequence: the 64 angles of the block's first row
// are reduced in fp64 once (shared memory), each row adds its offset's angle in
// fp32; 16-byte loads and stores, one pass over x.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "rope.cuh"

namespace yoco {

template <typename T, int D>
__global__ void __launch_bounds__(256) rope_apply_kernel(T *x, int N, int H, int64_t pos0, float base) {
    constexpr int EV = 16 / sizeof(T);      // elements per 16-byte chunk (an even number)
    constexpr int CH = D / EV;              // chunks per head row
    __shared__ float bc[D / 2], bs[D / 2], th[D / 2];
    const int n0 = blockIdx.x * 128, b = blockIdx.y;
    if (threadIdx.x < D / 2) {
        const double t = rope_theta(threadIdx.x, D, base);
        rope_cs_exact(pos0 + n0, t, bc[threadIdx.x], bs[threadIdx.x]);
        th[threadIdx.x] = (float)t;
    }
    __syncthreads();
    const int rows = min(128, N - n0);
    const int64_t total = (int64_t)rows * H * CH;
    for (int64_t e = threadIdx.x; e < total; e += blockDim.x) {
        const int ch = (int)(e % CH);
        const int64_t rh = e / CH;
        const int h = (int)(rh % H), j = (int)(rh / H);
        T *p = x + (((size_t)b * N + n0 + j) * H + h) * D + (size_t)ch * EV;
        uint4 u = *reinterpret_cast<const uint4 *>(p);
        if constexpr (sizeof(T) == 2) {
            uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int i = ch * 4 + q;
                float x0 = __uint_as_float(w[q] << 16), x1 = __uint_as_float(w[q] & 0xFFFF0000u);
                float cj, sj, c, s;
                rope_cs_offset(j, th[i], cj, sj);
                rope_cs_add(bc[i], bs[i], cj, sj, c, s);
                rope_turn(x0, x1, c, s);
                __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
                w[q] = *reinterpret_cast<uint32_t *>(&h2);
            }
            u = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            float f[4] = {__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w)};
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int i = ch * 2 + q;
                float cj, sj, c, s;
                rope_cs_offset(j, th[i], cj, sj);
                rope_cs_add(bc[i], bs[i], cj, sj, c, s);
                rope_turn(f[2 * q], f[2 * q + 1], c, s);
            }
            u = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
        }
        *reinterpret_cast<uint4 *>(p) = u;
    }
}

}  // namespace yoco

namespace yoco_host {
using namespace yoco;

cudaError_t rope_apply(void *x, int B, int N, int H, int d, int64_t pos0, float base, yoco_dtype dt, cudaStream_t st) {
    if (N <= 0) return cudaSuccess;
    dim3 grid((N + 127) / 128, B);
    count_launches(1);
    if (dt == YOCO_BF16) {
        if (d == 128) rope_apply_kernel<bf16_t, 128><<<grid, 256, 0, st>>>((bf16_t *)x, N, H, pos0, base);
        else rope_apply_kernel<bf16_t, 64><<<grid, 256, 0, st>>>((bf16_t *)x, N, H, pos0, base);
    } else {
        if (d == 128) rope_apply_kernel<float, 128><<<grid, 256, 0, st>>>((float *)x, N, H, pos0, base);
        else rope_apply_kernel<float, 64><<<grid, 256, 0, st>>>((float *)x, N, H, pos0, base);
    }
    return cudaGetLastError();
}

}  // namespace yoco_host
