// rope.cu -- rotary position encoding of token-major q or k in place (paper
// Section 3.1: Q (.) Theta, K (.) conj(Theta); the gRet and sliding-window
// self-decoders rotate their own q and k before their token mixer).  Channel pair
// (2i, 2i+1) of row n (every head, every sequence) turns by (pos0 + n) theta_i.
//
// One CTA per 32 rows of one sequence: the angles of the block's first row are
// reduced in fp64 once per thread's pairs, each row adds its offset's angle in
// fp32; 16-byte loads and stores, one pass over x.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "rope.cuh"

namespace yoco {

// Thread = one 16-byte chunk position of a head row (fixed pairs i), looping over
// the block's rows and heads with 32-bit indices, four items' loads issued before
// their arithmetic: the chunk's base angles and frequencies stay in registers.
constexpr int kRopeRows = 32;  // rows per CTA of rope_apply_kernel

template <typename T, int D>
__global__ void __launch_bounds__(256) rope_apply_kernel(T *x, int N, int H, int64_t pos0, const RopeFreq rf) {
    constexpr int EV = 16 / sizeof(T);      // elements per 16-byte chunk (an even number)
    constexpr int PC = EV / 2;              // pairs per chunk
    constexpr int CH = D / EV;              // chunks per head row
    constexpr int STEP = 256 / CH;          // (row, head) items a CTA pass covers
    const int n0 = blockIdx.x * kRopeRows, b = blockIdx.y;
    const int ch = threadIdx.x % CH;
    float bc[PC], bs[PC], th[PC];
#pragma unroll
    for (int q = 0; q < PC; ++q) {
        rope_cs_exact(pos0 + n0, rf.theta[ch * PC + q], bc[q], bs[q]);
        th[q] = (float)rf.theta[ch * PC + q];
    }
    const int rows = min(kRopeRows, N - n0);
    const int items = rows * H;
    if (!YOCO_DCHECK(n0 < N && b < (int)gridDim.y, 0x5D)) return;
    T *xb = x + ((size_t)b * N + n0) * H * D + ch * EV;
    constexpr int U = 4;  // items of a thread in flight at once, loads first
    for (int it0 = threadIdx.x / CH; it0 < items; it0 += U * STEP) {
        uint4 uu[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int it = it0 + k * STEP;
            if (it < items) uu[k] = *reinterpret_cast<const uint4 *>(xb + (size_t)it * D);
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int it = it0 + k * STEP;
            if (it >= items) break;
            const int j = it / H;  // row offset inside the block (item = j * H + h)
            uint4 u = uu[k];
            float c[PC], s[PC];
#pragma unroll
            for (int q = 0; q < PC; ++q) {
                float cj, sj;
                rope_cs_offset(j, th[q], cj, sj);
                rope_cs_add(bc[q], bs[q], cj, sj, c[q], s[q]);
            }
            if constexpr (sizeof(T) == 2) {
                uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float x0 = __uint_as_float(w[q] << 16), x1 = __uint_as_float(w[q] & 0xFFFF0000u);
                    rope_turn(x0, x1, c[q], s[q]);
                    __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
                    w[q] = *reinterpret_cast<uint32_t *>(&h2);
                }
                u = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
                float f[4] = {__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w)};
#pragma unroll
                for (int q = 0; q < 2; ++q) rope_turn(f[2 * q], f[2 * q + 1], c[q], s[q]);
                u = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
            }
            *reinterpret_cast<uint4 *>(xb + (size_t)it * D) = u;
        }
    }
}

// (cos, sin) of (pos0 + t) theta_i for t < T, i < d/2 into tab[t][i]: one CTA per 128
// positions, the base angles in fp64 once, the offsets in fp32
__global__ void __launch_bounds__(256) rope_table_kernel(float2 *tab, int64_t pos0, int T, int half_d, const RopeFreq rf) {
    __shared__ float bc[64], bs[64], th[64];
    const int t0 = blockIdx.x * 128;
    if (threadIdx.x < half_d) {
        rope_cs_exact(pos0 + t0, rf.theta[threadIdx.x], bc[threadIdx.x], bs[threadIdx.x]);
        th[threadIdx.x] = (float)rf.theta[threadIdx.x];
    }
    __syncthreads();
    const int rows = min(128, T - t0);
    for (int e = threadIdx.x; e < rows * half_d; e += blockDim.x) {
        const int j = e / half_d, i = e % half_d;
        float cj, sj, c, s;
        rope_cs_offset(j, th[i], cj, sj);
        rope_cs_add(bc[i], bs[i], cj, sj, c, s);
        tab[(size_t)(t0 + j) * half_d + i] = make_float2(c, s);
    }
}

}  // namespace yoco

namespace yoco_host {
using namespace yoco;

cudaError_t rope_apply(void *x, int B, int N, int H, int d, int64_t pos0, float base, yoco_dtype dt, cudaStream_t st) {
    if (N <= 0) return cudaSuccess;
    dim3 grid((N + kRopeRows - 1) / kRopeRows, B);
    const RopeFreq rf = make_rope_freq(base, d);
    count_launches(1);
    if (dt == YOCO_BF16) {
        if (d == 128) rope_apply_kernel<bf16_t, 128><<<grid, 256, 0, st>>>((bf16_t *)x, N, H, pos0, rf);
        else rope_apply_kernel<bf16_t, 64><<<grid, 256, 0, st>>>((bf16_t *)x, N, H, pos0, rf);
    } else {
        if (d == 128) rope_apply_kernel<float, 128><<<grid, 256, 0, st>>>((float *)x, N, H, pos0, rf);
        else rope_apply_kernel<float, 64><<<grid, 256, 0, st>>>((float *)x, N, H, pos0, rf);
    }
    return cudaGetLastError();
}

cudaError_t rope_table(float2 *tab, int64_t pos0, int T, int d, float base, cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    count_launches(1);
    rope_table_kernel<<<(T + 127) / 128, 256, 0, st>>>(tab, pos0, T, d / 2, make_rope_freq(base, d));
    return cudaGetLastError();
}

}  // namespace yoco_host

YOCO_DEBUG_TU(rope)
