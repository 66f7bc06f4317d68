// kv_proj.cu -- shared K^/V^ projection fused with RMSNorm and the cache append
// (paper Section 2.2, Eq. 2: K^ = LN(M) W_K, V^ = LN(M) W_V with LN = RMSNorm).
//
// RMSNorm is applied as a row scale after the product: RMSNorm(m) W = r (m * g) W
// with r = 1 / sqrt(mean(m^2) + eps), so the GEMM runs on the raw rows and the
// per-row r (one warp per row, fp32) multiplies the fp32 accumulator in the
// epilogue, which rounds once to the cache type and scatters each row into slot
// len + t of every kv head.  The last CTA to finish advances the device length.
//
// This file holds the CUDA-core path (any dtype, any T); large bf16 appends go to
// the tensor-core GEMM in kv_proj_tc.cu.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace yoco {

// r_row = 1 / sqrt(mean(M_row^2) + eps), one warp per row
template <typename T>
__global__ void rms_rows_kernel(const T *__restrict__ M, float *__restrict__ r, int rows, int dm, float eps) {
    const int w = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
    const int lane = threadIdx.x % 32;
    if (w >= rows) return;
    const T *row = M + (size_t)w * dm;
    float ss = 0.f;
    for (int i = lane; i < dm; i += 32) {
        float x = to_f32(row[i]);
        ss = fmaf(x, x, ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane == 0) r[w] = rsqrtf(ss / (float)dm + eps);
}

// Marks one CTA done; the last one publishes len + T.  len_dev[1] counts CTAs and
// is reset to 0 by the last one, ready for the next append.
__device__ __forceinline__ void finish_append(int32_t *len_dev, int64_t new_len) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned total = gridDim.x * gridDim.y * gridDim.z;
        unsigned ticket = atomicAdd(reinterpret_cast<unsigned *>(len_dev + 1), 1u);
        if (ticket == total - 1) {
            len_dev[0] = (int32_t)new_len;
            __threadfence();
            atomicExch(reinterpret_cast<unsigned *>(len_dev + 1), 0u);
        }
    }
}

// out[R, 2n] = (M * g)[R, dm] @ [Wk | Wv][dm, 2n], scaled by r per row, into the cache.
// 64 x 64 tile per CTA, 256 threads x (4 x 4) outputs, fp32 accumulate.
template <typename T>
__global__ void __launch_bounds__(256)
proj_append_simt(const T *__restrict__ M, const T *__restrict__ g, const T *__restrict__ Wk,
                 const T *__restrict__ Wv, const float *__restrict__ r, T *__restrict__ kc, T *__restrict__ vc,
                 int R, int T_rows, int dm, int Hkv, int d, int64_t cap, int64_t len, int32_t *len_dev) {
    constexpr int BM = 64, BN = 64, BK = 16;
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    const int n = Hkv * d;
    const int row0 = blockIdx.y * BM, col0 = blockIdx.x * BN;  // col in [0, 2n)
    const int tid = threadIdx.x;
    const int tr = tid / 16, tc = tid % 16;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < dm; k0 += BK) {
        for (int e = tid; e < BM * BK; e += 256) {
            int rr = e / BK, kk = e % BK;
            int row = row0 + rr, kx = k0 + kk;
            float x = 0.f;
            if (row < R && kx < dm) {
                x = to_f32(M[(size_t)row * dm + kx]);
                if (g) x *= to_f32(g[kx]);
            }
            As[kk][rr] = x;
        }
        for (int e = tid; e < BK * BN; e += 256) {
            int kk = e / BN, cc = e % BN;
            int col = col0 + cc, kx = k0 + kk;
            float w = 0.f;
            if (col < 2 * n && kx < dm) {
                const T *W = (col < n) ? Wk : Wv;
                w = to_f32(W[(size_t)kx * n + (col % n)]);
            }
            Bs[kk][cc] = w;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[4], bb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = As[kk][tr * 4 + i];
                bb[i] = Bs[kk][tc * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int row = row0 + tr * 4 + i;
        if (row >= R) continue;
        int b = row / T_rows, t = row % T_rows;
        float rs = r[row];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int col = col0 + tc * 4 + j;
            if (col >= 2 * n) continue;
            int cn = col % n, h = cn / d, c = cn % d;
            T *dst = (col < n) ? kc : vc;
            dst[(((size_t)b * Hkv + h) * cap + len + t) * d + c] = from_f32<T>(acc[i][j] * rs);
        }
    }
    finish_append(len_dev, len + T_rows);
}

// Few rows (decode): split-K GEMV.  CTA (column group, K slice) of 256 threads;
// thread = 8 consecutive output columns (one 16-byte row segment of W), looping
// over its slice of W rows and over the input rows 4 at a time; fp32 partials
// go to the workspace and proj_gemv_finish sums them.
template <typename T>
__global__ void __launch_bounds__(256)
proj_gemv_partial(const T *__restrict__ M, const T *__restrict__ g, const T *__restrict__ Wk,
                  const T *__restrict__ Wv, float *__restrict__ part, int R, int dm, int n, int rows_per_split) {
    const int col = (blockIdx.x * 256 + threadIdx.x) * 8;  // in [0, 2n)
    const int k0 = blockIdx.y * rows_per_split;
    const int k1 = min(dm, k0 + rows_per_split);
    extern __shared__ float msh[];  // [R][rows_per_split]
    for (int e = threadIdx.x; e < R * rows_per_split; e += 256) {
        int r = e / rows_per_split, kk = k0 + e % rows_per_split;
        float x = 0.f;
        if (kk < k1) {
            x = to_f32(M[(size_t)r * dm + kk]);
            if (g) x *= to_f32(g[kk]);
        }
        msh[e] = x;
    }
    __syncthreads();
    if (col >= 2 * n) return;
    const T *W = (col < n) ? Wk : Wv;
    const int wc = col % n;
    for (int r0 = 0; r0 < R; r0 += 4) {
        float acc[4][8] = {};
        for (int kk = k0; kk < k1; ++kk) {
            float w[8];
            if constexpr (sizeof(T) == 2) {
                uint4 u = *reinterpret_cast<const uint4 *>(W + (size_t)kk * n + wc);
                uint32_t x[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    w[2 * e] = __uint_as_float(x[e] << 16);
                    w[2 * e + 1] = __uint_as_float(x[e] & 0xFFFF0000u);
                }
            } else {
                const float4 *p = reinterpret_cast<const float4 *>(W + (size_t)kk * n + wc);
                float4 a = p[0], b = p[1];
                w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
            }
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const float m = (r0 + rr < R) ? msh[(r0 + rr) * rows_per_split + (kk - k0)] : 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[rr][e] = fmaf(m, w[e], acc[rr][e]);
            }
        }
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            if (r0 + rr >= R) break;
            float4 *dst = reinterpret_cast<float4 *>(part + ((size_t)blockIdx.y * R + r0 + rr) * 2 * n + col);
            dst[0] = make_float4(acc[rr][0], acc[rr][1], acc[rr][2], acc[rr][3]);
            dst[1] = make_float4(acc[rr][4], acc[rr][5], acc[rr][6], acc[rr][7]);
        }
    }
}

// sum the K slices, apply the RMS factor, round once, write the cache slot
template <typename T>
__global__ void proj_gemv_finish(const float *__restrict__ part, const float *__restrict__ r, T *__restrict__ kc,
                                 T *__restrict__ vc, int R, int T_rows, int n, int Hkv, int d, int64_t cap,
                                 int64_t len, int splits, int32_t *len_dev) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;  // over R * 2n
    if (idx < R * 2 * n) {
        const int row = idx / (2 * n), col = idx % (2 * n);
        float acc = 0.f;
        for (int s = 0; s < splits; ++s) acc += part[((size_t)s * R + row) * 2 * n + col];
        const int b = row / T_rows, t = row % T_rows;
        const int cn = col % n, h = cn / d, c = cn % d;
        T *dst = (col < n) ? kc : vc;
        dst[(((size_t)b * Hkv + h) * cap + len + t) * d + c] = from_f32<T>(acc * r[row]);
    }
    finish_append(len_dev, len + T_rows);
}

}  // namespace yoco

namespace yoco_host {
using namespace yoco;

constexpr int kGemvMaxRows = 16;
constexpr int kGemvSplits = 128;

static bool gemv_eligible(int R, int n) { return R <= kGemvMaxRows && n % 8 == 0; }

// workspace: [0, 256) status word of the tensor-core kernel, one fp32 RMS factor
// per row, then (few-row path) the split-K partials
size_t kv_proj_workspace(int B, int T, int dm, int Hkv, int d, yoco_dtype dt) {
    (void)dm; (void)dt;
    size_t rows = (size_t)B * T;
    size_t ws = 256 + ((rows * sizeof(float) + 255) / 256) * 256;
    const int n = Hkv * d;
    if (gemv_eligible((int)rows, n)) ws += (size_t)kGemvSplits * rows * 2 * n * sizeof(float);
    return ws;
}

template <typename T>
static cudaError_t run(const KvProjArgs &a, void *ws, cudaStream_t st) {
    const int R = a.B * a.T;
    float *r = (float *)((char *)ws + 256);
    count_launches(1);
    rms_rows_kernel<T><<<(R * 32 + 255) / 256, 256, 0, st>>>((const T *)a.M, r, R, a.dm, a.eps);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (std::is_same<T, bf16_t>::value && kv_proj_tc_eligible(a)) return kv_project_append_tc(a, r, (int *)ws, st);
    const int n = a.Hkv * a.d;
    if (gemv_eligible(R, n)) {
        float *part = r + ((size_t)R + 63) / 64 * 64;
        const int rows_per_split = (a.dm + kGemvSplits - 1) / kGemvSplits;
        const int splits = (a.dm + rows_per_split - 1) / rows_per_split;
        dim3 g1((2 * n / 8 + 255) / 256, splits);
        count_launches(2);
        proj_gemv_partial<T><<<g1, 256, (size_t)R * rows_per_split * sizeof(float), st>>>(
            (const T *)a.M, (const T *)a.rms_w, (const T *)a.Wk, (const T *)a.Wv, part, R, a.dm, n, rows_per_split);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        const int total = R * 2 * n;
        proj_gemv_finish<T><<<(total + 255) / 256, 256, 0, st>>>(part, r, (T *)a.kc, (T *)a.vc, R, a.T, n, a.Hkv, a.d,
                                                                 a.cap, a.len, splits, a.len_dev);
        return cudaGetLastError();
    }
    count_launches(1);
    dim3 grid((2 * a.Hkv * a.d + 63) / 64, (R + 63) / 64);
    proj_append_simt<T><<<grid, 256, 0, st>>>((const T *)a.M, (const T *)a.rms_w, (const T *)a.Wk, (const T *)a.Wv,
                                              r, (T *)a.kc, (T *)a.vc, R, a.T, a.dm, a.Hkv, a.d, a.cap, a.len,
                                              a.len_dev);
    return cudaGetLastError();
}

cudaError_t kv_project_append(const KvProjArgs &a, void *ws, cudaStream_t st) {
    if (a.dt == YOCO_BF16) return run<bf16_t>(a, ws, st);
    return run<float>(a, ws, st);
}

}  // namespace yoco_host
