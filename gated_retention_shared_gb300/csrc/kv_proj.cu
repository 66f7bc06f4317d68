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
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "rope.cuh"

namespace yoco {

// r_row = 1 / sqrt(mean(M_row^2) + eps), one warp per row (rows strided over a
// grid of at most one wave, 16-byte loads when the rows allow).  It releases its
// programmatic dependents at once, so the tensor-core GEMM that follows is
// launched while it runs; the GEMM's CTAs find room on an SM only as this pass's
// CTAs leave it (eight of them fill an SM's threads), so the two run one after
// the other, without a launch gap.  Measured on the 512K-row projection, running
// this pass beside the GEMM (one small CTA per SM, per-row-group ready flags) made
// the GEMM slower by about the pass's own time, and summing the squares inside
// the GEMM from its staged tiles slowed its pipeline more than the pass costs.
template <typename T>
__global__ void rms_rows_kernel(const T *__restrict__ M, float *__restrict__ r, int rows, int dm, float eps) {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    constexpr int EV = 16 / sizeof(T);  // elements per 16-byte load
    const int lane = threadIdx.x % 32;
    const int warps = gridDim.x * (blockDim.x / 32);
    const bool vec = (dm % EV) == 0;
    for (int w = (blockIdx.x * blockDim.x + threadIdx.x) / 32; w < rows; w += warps) {
        const T *row = M + (size_t)w * dm;
        float ss = 0.f;
        if (vec) {
            for (int i = lane * EV; i < dm; i += 32 * EV) {
                const uint4 u = *reinterpret_cast<const uint4 *>(row + i);
                if constexpr (sizeof(T) == 2) {
                    const uint32_t x[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float lo = __uint_as_float(x[e] << 16), hi = __uint_as_float(x[e] & 0xFFFF0000u);
                        ss = fmaf(lo, lo, ss);
                        ss = fmaf(hi, hi, ss);
                    }
                } else {
                    const float f[4] = {__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                                        __uint_as_float(u.w)};
#pragma unroll
                    for (int e = 0; e < 4; ++e) ss = fmaf(f[e], f[e], ss);
                }
            }
        } else {
            for (int i = lane; i < dm; i += 32) {
                const float x = to_f32(row[i]);
                ss = fmaf(x, x, ss);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (lane == 0) r[w] = rsqrtf(ss / (float)dm + eps);
    }
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
                 int R, int T_rows, int dm, int Hkv, int d, int64_t cap, int64_t len, int32_t *len_dev,
                 float rope_base, const RopeFreq rf) {
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
        float val[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) val[j] = acc[i][j] * rs;
        // the thread's 4 columns lie in one head of Wk or Wv (d, n multiples of 64)
        const int col4 = col0 + tc * 4;
        if (rope_base > 0.f && col4 < n) {  // rotary encoding of K^ at slot position len + t
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float cs, sn;
                rope_cs_exact(len + t, rf.theta[(col4 % d) / 2 + q], cs, sn);
                rope_turn(val[2 * q], val[2 * q + 1], cs, sn);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int col = col4 + j;
            if (col >= 2 * n) continue;
            int cn = col % n, h = cn / d, c = cn % d;
            T *dst = (col < n) ? kc : vc;
            if (YOCO_DCHECK(len + t < cap && h < Hkv, 0x4A))
                dst[(((size_t)b * Hkv + h) * cap + len + t) * d + c] = from_f32<T>(val[j]);
        }
    }
    finish_append(len_dev, len + T_rows);
}

// Few rows (decode): one GEMV launch, split over K.  CTA (column group cg, K
// chunk kc), 256 threads = 8 warps: lane l owns the 8 columns cg * 256 + 8 l
// (one 16-byte W segment, so a warp reads 512 contiguous bytes of a W row), warp
// w the rows kc * KR + w, + 8, ... of the chunk.  The CTA sums its 8 warps in
// shared memory and writes one fp32 partial per (row, column) to the workspace;
// the last CTA to finish (ticket in len_dev[1], no waiting) adds the KCH partials
// in chunk order, computes each input row's RMS factor, rounds once, writes the
// cache slots and publishes the new length.
constexpr int kGemvU = 10;      // W rows in flight per warp (fp32 W; bf16 W: twice as many)
constexpr int kTailBatch = 10;  // K-chunk partials in flight per thread in the last CTA

// 8 consecutive W elements as raw 16-byte words (bf16: one, fp32: two)
template <typename T>
struct W8 {
    uint4 u[sizeof(T) / 2];
};
template <typename T>
__device__ __forceinline__ W8<T> ld_w8(const T *p) {
    W8<T> r;
#pragma unroll
    for (int i = 0; i < (int)(sizeof(T) / 2); ++i) r.u[i] = __ldg(reinterpret_cast<const uint4 *>(p) + i);
    return r;
}
template <typename T>
__device__ __forceinline__ void cvt_w8(const W8<T> &r, float w[8]) {
    if constexpr (sizeof(T) == 2) {
        const uint32_t x[4] = {r.u[0].x, r.u[0].y, r.u[0].z, r.u[0].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            w[2 * e] = __uint_as_float(x[e] << 16);
            w[2 * e + 1] = __uint_as_float(x[e] & 0xFFFF0000u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            w[4 * i] = __uint_as_float(r.u[i].x);
            w[4 * i + 1] = __uint_as_float(r.u[i].y);
            w[4 * i + 2] = __uint_as_float(r.u[i].z);
            w[4 * i + 3] = __uint_as_float(r.u[i].w);
        }
    }
}

template <typename T>
__device__ __forceinline__ void load_w8(const T *p, float w[8]) {
    if constexpr (sizeof(T) == 2) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
        const uint32_t x[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            w[2 * e] = __uint_as_float(x[e] << 16);
            w[2 * e + 1] = __uint_as_float(x[e] & 0xFFFF0000u);
        }
    } else {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p)), b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    }
}

template <typename T, int kGemvRG>
__global__ void __launch_bounds__(256)
proj_gemv_splitk(const T *__restrict__ M, const T *__restrict__ g, const T *__restrict__ Wk, const T *__restrict__ Wv,
                 float *__restrict__ part, T *__restrict__ kc, T *__restrict__ vc, int R, int T_rows, int dm, int n,
                 int Hkv, int d, int64_t cap, int64_t len, float eps, int KR, int32_t *len_dev, float rope_base,
                 const RopeFreq rf) {
    extern __shared__ float msh[];  // [kGemvRG][KR]: this chunk of the input rows, times the gain
    __shared__ float red[8][256];   // [warp][lane * 8 + e] for one input row
    __shared__ int last;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int col = blockIdx.x * 256 + lane * 8;  // first of this lane's 8 columns, in [0, 2n)
    const bool col_ok = col < 2 * n;
    const T *W = (col < n) ? Wk + col : Wv + (col - n);
    const int k0 = blockIdx.y * KR, k1 = min(dm, k0 + KR);
    const int nkc = gridDim.y;
    for (int r0 = 0; r0 < R; r0 += kGemvRG) {
        const int rg = min(kGemvRG, R - r0);
        for (int e = tid; e < rg * KR; e += 256) {
            const int rr = e / KR, kk = k0 + e % KR;
            float x = 0.f;
            if (kk < k1) {
                x = to_f32(M[(size_t)(r0 + rr) * dm + kk]);
                if (g) x *= to_f32(g[kk]);
            }
            msh[e] = x;
        }
        __syncthreads();
        float acc[kGemvRG][8] = {};
        auto fma_row = [&](const W8<T> &raw, int kk) {
            float w[8];
            cvt_w8(raw, w);
#pragma unroll
            for (int rr = 0; rr < kGemvRG; ++rr) {
                const float m = (rr < rg) ? msh[rr * KR + (kk - k0)] : 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[rr][e] = fmaf(m, w[e], acc[rr][e]);
            }
        };
        if (col_ok) {
            int kk = k0 + warp;
            // batches of U rows: every load of a batch is issued before its FMAs
            constexpr int U = (sizeof(T) == 2) ? 2 * kGemvU : kGemvU;
            for (; kk + 8 * (U - 1) < k1; kk += 8 * U) {
                W8<T> raw[U];
#pragma unroll
                for (int u = 0; u < U; ++u) raw[u] = ld_w8(W + (size_t)(kk + 8 * u) * n);
#pragma unroll
                for (int u = 0; u < U; ++u) fma_row(raw[u], kk + 8 * u);
            }
            for (; kk < k1; kk += 8) fma_row(ld_w8(W + (size_t)kk * n), kk);
        }
        for (int rr = 0; rr < rg; ++rr) {
#pragma unroll
            for (int e = 0; e < 8; ++e) red[warp][lane * 8 + e] = acc[rr][e];
            __syncthreads();
            // thread tid sums column tid of this group over the 8 warps
            const int c = blockIdx.x * 256 + tid;
            if (c < 2 * n) {
                float sum = 0.f;
#pragma unroll
                for (int w8 = 0; w8 < 8; ++w8) sum += red[w8][tid];
                part[((size_t)blockIdx.y * R + r0 + rr) * 2 * n + c] = sum;
            }
            __syncthreads();
        }
    }
    // the last CTA adds the chunks' partials (fixed order) and writes the slots
    __threadfence();  // this thread's partials are visible before the ticket is taken
    __syncthreads();
    if (tid == 0) {
        const unsigned total = gridDim.x * gridDim.y;
        last = (atomicAdd(reinterpret_cast<unsigned *>(len_dev + 1), 1u) == total - 1);
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    // Per row: the RMS factor of the raw input row and the sum of the K chunks'
    // partials for this thread's 8 columns.  Loads are issued in batches
    // (kTailBatch chunks at a time, the first batch together with the row's RMS
    // loads) so the tail costs a few L2 round trips, not one per chunk.
    const size_t qstride = (size_t)R * 2 * n;
    for (int row = 0; row < R; ++row) {
        const int b = row / T_rows, t = row % T_rows;
        float rms_r = 0.f;
        for (int c = tid * 8, first = 1; c < 2 * n || first; c += 256 * 8, first = 0) {
            const bool has_c = c < 2 * n;
            const float *pc = part + (size_t)row * 2 * n + (has_c ? c : 0);
            float sum[8] = {};
            auto add_batch = [&](int q0) {
                float4 v[kTailBatch][2];
#pragma unroll
                for (int u = 0; u < kTailBatch; ++u) {
                    if (q0 + u < nkc) {
                        v[u][0] = __ldcg(reinterpret_cast<const float4 *>(pc + (q0 + u) * qstride));
                        v[u][1] = __ldcg(reinterpret_cast<const float4 *>(pc + (q0 + u) * qstride) + 1);
                    } else {
                        v[u][0] = v[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
#pragma unroll
                for (int u = 0; u < kTailBatch; ++u) {
                    sum[0] += v[u][0].x; sum[1] += v[u][0].y; sum[2] += v[u][0].z; sum[3] += v[u][0].w;
                    sum[4] += v[u][1].x; sum[5] += v[u][1].y; sum[6] += v[u][1].z; sum[7] += v[u][1].w;
                }
            };
            if (first) {
                // the first batch of partials and the row's RMS loads in flight together
                float4 v0[kTailBatch][2];
                if (has_c) {
#pragma unroll
                    for (int u = 0; u < kTailBatch; ++u) {
                        if (u < nkc) {
                            v0[u][0] = __ldcg(reinterpret_cast<const float4 *>(pc + u * qstride));
                            v0[u][1] = __ldcg(reinterpret_cast<const float4 *>(pc + u * qstride) + 1);
                        } else {
                            v0[u][0] = v0[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                    }
                }
                float ss = 0.f;
#pragma unroll 4
                for (int kv = tid * 8; kv < dm; kv += 256 * 8) {
                    float x[8];
                    load_w8(M + (size_t)row * dm + kv, x);
#pragma unroll
                    for (int q = 0; q < 8; ++q) ss = fmaf(x[q], x[q], ss);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                if (lane == 0) red[0][warp] = ss;
                __syncthreads();
                float sq = 0.f;
#pragma unroll
                for (int w8 = 0; w8 < 8; ++w8) sq += red[0][w8];
                rms_r = rsqrtf(sq / (float)dm + eps);
                if (has_c) {
#pragma unroll
                    for (int u = 0; u < kTailBatch; ++u) {
                        sum[0] += v0[u][0].x; sum[1] += v0[u][0].y; sum[2] += v0[u][0].z; sum[3] += v0[u][0].w;
                        sum[4] += v0[u][1].x; sum[5] += v0[u][1].y; sum[6] += v0[u][1].z; sum[7] += v0[u][1].w;
                    }
                }
            }
            if (!has_c) continue;
            for (int q0 = first ? kTailBatch : 0; q0 < nkc; q0 += kTailBatch) add_batch(q0);
            // the 8 columns lie in one head of Wk or of Wv (n % 8 == 0, d % 8 == 0)
            const int cn = c % n, h = cn / d, cc = cn % d;
            if (!YOCO_DCHECK(len + t < cap && h < Hkv && cc + 8 <= d, 0x49)) continue;
            T *dst = ((c < n) ? kc : vc) + (((size_t)b * Hkv + h) * cap + len + t) * d + cc;
#pragma unroll
            for (int e = 0; e < 8; ++e) sum[e] *= rms_r;
            if (rope_base > 0.f && c < n) {  // rotary encoding of K^ at slot position len + t
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float cs, sn;
                    rope_cs_exact(len + t, rf.theta[cc / 2 + q], cs, sn);
                    rope_turn(sum[2 * q], sum[2 * q + 1], cs, sn);
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) dst[e] = from_f32<T>(sum[e]);
        }
        __syncthreads();  // red[0] is rewritten for the next row
    }
    if (tid == 0) {
        len_dev[0] = (int32_t)(len + T_rows);
        __threadfence();
        atomicExch(reinterpret_cast<unsigned *>(len_dev + 1), 0u);
    }
}

// Few rows, bf16 (decode): column strips.  CTA = 16 output columns of [W_K | W_V]
// over the whole of d_model, 512 threads.  Lanes 2r and 2r + 1 of a warp read the
// two 16-byte halves of one W row's 32-byte strip (one sector), so a warp's load
// takes 16 whole sectors and every W byte is read once, by one CTA, in one round
// of loads issued before the wait on the previous kernel (the weights are not
// written by it; the input rows M may be).  Thread t covers rows t / 2, t / 2 + 256,
// ... and columns 8 (t % 2) .. + 7 of the strip.  The products, and each input row's
// sum of squares for the RMS factor, are reduced inside the CTA by warp shuffles
// and one pass through shared memory: no partial sums leave the CTA and no CTA
// waits for another.
constexpr int kStripThreads = 512;
constexpr int kStripCols = 16;
constexpr int kStripRowsPerPass = kStripThreads / 2;  // W rows one round of loads covers

template <int KR, int RG>
__global__ void __launch_bounds__(kStripThreads, 1)
proj_gemv_strip(const bf16_t *__restrict__ M, const bf16_t *__restrict__ g, const bf16_t *__restrict__ Wk,
                const bf16_t *__restrict__ Wv, bf16_t *__restrict__ kc, bf16_t *__restrict__ vc, int R, int T_rows,
                int dm, int n, int Hkv, int d, int64_t cap, int64_t len, float eps, int32_t *len_dev,
                float rope_base, const RopeFreq rf) {
    __shared__ float red[kStripThreads / 32][RG][kStripCols + 1];  // per warp: 16 column sums, sum of squares
    __shared__ float fin[RG][kStripCols + 1];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int half = tid & 1;                              // columns 8 half .. 8 half + 7 of the strip
    const int c0 = blockIdx.x * kStripCols;               // first column of the strip in [0, 2n)
    const bf16_t *W = ((c0 < n) ? Wk + c0 : Wv + (c0 - n)) + 8 * half;  // n % 16 == 0: the strip lies in one
    uint4 wr[KR];
#pragma unroll
    for (int i = 0; i < KR; ++i) {
        const int k = (tid >> 1) + i * kStripRowsPerPass;
        wr[i] = (k < dm) ? __ldg(reinterpret_cast<const uint4 *>(W + (size_t)k * n)) : make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("griddepcontrol.wait;\n" ::: "memory");  // M (and the cache) after the previous kernel
    for (int r0 = 0; r0 < R; r0 += RG) {
        float acc[RG][8], ss[RG];
#pragma unroll
        for (int rr = 0; rr < RG; ++rr) {
            ss[rr] = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[rr][e] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < KR; ++i) {
            const int k = (tid >> 1) + i * kStripRowsPerPass;
            if (k >= dm) continue;
            float w[8];
            const uint32_t x[4] = {wr[i].x, wr[i].y, wr[i].z, wr[i].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                w[2 * e] = __uint_as_float(x[e] << 16);
                w[2 * e + 1] = __uint_as_float(x[e] & 0xFFFF0000u);
            }
            const float gk = g ? to_f32(g[k]) : 1.f;
#pragma unroll
            for (int rr = 0; rr < RG; ++rr) {
                if (r0 + rr >= R) break;
                const float m = to_f32(M[(size_t)(r0 + rr) * dm + k]);
                if (half == 0) ss[rr] = fmaf(m, m, ss[rr]);  // each row's squares once
                const float mg = m * gk;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[rr][e] = fmaf(mg, w[e], acc[rr][e]);
            }
        }
        // lanes of one half hold the same 8 columns: add over lanes 2 apart and more
#pragma unroll
        for (int rr = 0; rr < RG; ++rr) {
#pragma unroll
            for (int off = 16; off > 1; off >>= 1) {
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[rr][e] += __shfl_xor_sync(0xffffffffu, acc[rr][e], off);
                ss[rr] += __shfl_xor_sync(0xffffffffu, ss[rr], off);
            }
            if (lane < 2) {  // lane = half
#pragma unroll
                for (int e = 0; e < 8; ++e) red[warp][rr][8 * lane + e] = acc[rr][e];
                if (lane == 0) red[warp][rr][kStripCols] = ss[rr];
            }
        }
        __syncthreads();
        if (tid < RG * (kStripCols + 1)) {  // (row, column or sum of squares): add the 16 warps in order
            const int rr = tid / (kStripCols + 1), e = tid % (kStripCols + 1);
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < kStripThreads / 32; ++w) sum += red[w][rr][e];
            fin[rr][e] = sum;
        }
        __syncthreads();
        if (tid < RG * (kStripCols / 2)) {  // one channel pair of one row: scale, rotate (K^), round, store
            const int rr = tid / (kStripCols / 2), j = tid % (kStripCols / 2), row = r0 + rr;
            if (row < R) {
                const int b = row / T_rows, t = row % T_rows;
                const float rms = rsqrtf(fin[rr][kStripCols] / (float)dm + eps);
                float x0 = fin[rr][2 * j] * rms, x1 = fin[rr][2 * j + 1] * rms;
                const int c = c0 + 2 * j, cn = c % n, h = cn / d, cc = cn % d;
                if (rope_base > 0.f && c < n) {  // rotary encoding of K^ at slot position len + t
                    float cs, sn;
                    rope_cs_exact(len + t, rf.theta[cc / 2], cs, sn);
                    rope_turn(x0, x1, cs, sn);
                }
                bf16_t *dst = ((c < n) ? kc : vc) + (((size_t)b * Hkv + h) * cap + len + t) * d + cc;
                if (YOCO_DCHECK(len + t < cap && h < Hkv && c + 2 <= 2 * n, 0x48)) {
                    dst[0] = from_f32<bf16_t>(x0);
                    dst[1] = from_f32<bf16_t>(x1);
                }
            }
        }
        __syncthreads();  // red and fin are rewritten by the next rows
    }
    // No kernel reads the length on the device, and this grid releases no dependent
    // early, so whatever runs next on the stream sees every slot and the new length:
    // one thread publishes it, no ticket needed.
    if (blockIdx.x == 0 && tid == 0) len_dev[0] = (int32_t)(len + T_rows);
}

}  // namespace yoco

namespace yoco_host {
using namespace yoco;

constexpr int kGemvMaxRows = 16;

static bool gemv_eligible(int R, int n, int dm) { return R <= kGemvMaxRows && n % 8 == 0 && dm % 8 == 0; }

// K chunks of the few-row path: about one CTA per SM over all column groups
static int gemv_chunks(int n, int dm) {
    const int groups = (2 * n + 255) / 256;
    int kch = std::max(1, device_sm_count() / groups);
    kch = std::min(kch, dm);
    const int kr = (dm + kch - 1) / kch;
    return (dm + kr - 1) / kr;
}

constexpr int kStripMaxRows = 4;

static bool strip_eligible(int R, int n, int dm, yoco_dtype dt) {
    return dt == YOCO_BF16 && R <= kStripMaxRows && n % kStripCols == 0 && dm % 8 == 0 && dm <= 12 * kStripRowsPerPass;
}

// workspace: [0, 256) status word of the tensor-core kernel, one fp32 RMS factor
// per row (tensor-core and tiled paths), then (few-row path) the K-chunk partials
// workspace: [0, 256) status word, one fp32 RMS factor per row (padded to 256 B), then
// either the few-row path's K-chunk partials or, with rotary encoding on the other
// paths, the (cos, sin) table of the T positions [T][d/2] (the paths never meet)
size_t kv_proj_workspace(int B, int T, int dm, int Hkv, int d, yoco_dtype dt, float rope_base) {
    size_t rows = (size_t)B * T;
    size_t ws = 256 + ((rows * sizeof(float) + 255) / 256) * 256;
    const int n = Hkv * d;
    size_t extra = 0;
    if (strip_eligible((int)rows, n, dm, dt)) extra = 0;
    else if (gemv_eligible((int)rows, n, dm)) extra = (size_t)gemv_chunks(n, dm) * rows * 2 * n * sizeof(float);
    else if (rope_base > 0.f) extra = (size_t)T * (d / 2) * sizeof(float2);
    return ws + extra;
}

template <int KR>
static cudaError_t launch_strip(const KvProjArgs &a, int R, int n, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * n / kStripCols);
    cfg.blockDim = dim3(kStripThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launches(1);
    const RopeFreq rf = make_rope_freq(a.rope_base, a.d);
    if (R == 1)
        return cudaLaunchKernelEx(&cfg, proj_gemv_strip<KR, 1>, (const bf16_t *)a.M, (const bf16_t *)a.rms_w,
                                  (const bf16_t *)a.Wk, (const bf16_t *)a.Wv, (bf16_t *)a.kc, (bf16_t *)a.vc, R, a.T,
                                  a.dm, n, a.Hkv, a.d, a.cap, a.len, a.eps, a.len_dev, a.rope_base, rf);
    return cudaLaunchKernelEx(&cfg, proj_gemv_strip<KR, 2>, (const bf16_t *)a.M, (const bf16_t *)a.rms_w,
                              (const bf16_t *)a.Wk, (const bf16_t *)a.Wv, (bf16_t *)a.kc, (bf16_t *)a.vc, R, a.T, a.dm,
                              n, a.Hkv, a.d, a.cap, a.len, a.eps, a.len_dev, a.rope_base, rf);
}

template <typename T>
static cudaError_t run(const KvProjArgs &a, void *ws, cudaStream_t st) {
    const int R = a.B * a.T;
    const int n = a.Hkv * a.d;
    float *r = (float *)((char *)ws + 256);
    cudaError_t e;
    if (strip_eligible(R, n, a.dm, a.dt)) {
        const int kr = (a.dm + kStripRowsPerPass - 1) / kStripRowsPerPass;  // W rows per thread
        if (kr <= 4) return launch_strip<4>(a, R, n, st);
        if (kr <= 8) return launch_strip<8>(a, R, n, st);
        return launch_strip<12>(a, R, n, st);
    }
    if (gemv_eligible(R, n, a.dm) && !(std::is_same<T, bf16_t>::value && kv_proj_tc_eligible(a))) {
        const int kch = gemv_chunks(n, a.dm);
        const int KR = (a.dm + kch - 1) / kch;
        const int rg = (R == 1) ? 1 : 4;  // input rows per pass
        const size_t smem = (size_t)rg * KR * sizeof(float);
        auto kern = (R == 1) ? proj_gemv_splitk<T, 1> : proj_gemv_splitk<T, 4>;
        if (smem > 48 * 1024 &&
            (e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        float *part = r + ((size_t)R + 63) / 64 * 64;
        count_launches(1);
        kern<<<dim3((2 * n + 255) / 256, kch), 256, smem, st>>>(
            (const T *)a.M, (const T *)a.rms_w, (const T *)a.Wk, (const T *)a.Wv, part, (T *)a.kc, (T *)a.vc, R, a.T,
            a.dm, n, a.Hkv, a.d, a.cap, a.len, a.eps, KR, a.len_dev, a.rope_base, make_rope_freq(a.rope_base, a.d));
        return cudaGetLastError();
    }
    const bool tc = std::is_same<T, bf16_t>::value && kv_proj_tc_eligible(a);
    float2 *rope_cs = nullptr;
    if (tc && a.rope_base > 0.f) {
        // the positions' (cos, sin) table for the GEMM epilogue, filled before the RMS pass
        // (that pass releases the GEMM early, and the GEMM waits for it only)
        rope_cs = reinterpret_cast<float2 *>(r + ((size_t)R + 63) / 64 * 64);
        if ((e = rope_table(rope_cs, a.len, a.T, a.d, a.rope_base, st)) != cudaSuccess) return e;
    }
    count_launches(1);
    rms_rows_kernel<T><<<std::min((R * 32 + 255) / 256, device_sm_count() * 8), 256, 0, st>>>((const T *)a.M, r, R, a.dm, a.eps);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (tc) return kv_project_append_tc(a, r, rope_cs, (int *)ws, st);
    count_launches(1);
    dim3 grid((2 * a.Hkv * a.d + 63) / 64, (R + 63) / 64);
    proj_append_simt<T><<<grid, 256, 0, st>>>((const T *)a.M, (const T *)a.rms_w, (const T *)a.Wk, (const T *)a.Wv,
                                              r, (T *)a.kc, (T *)a.vc, R, a.T, a.dm, a.Hkv, a.d, a.cap, a.len,
                                              a.len_dev, a.rope_base, make_rope_freq(a.rope_base, a.d));
    return cudaGetLastError();
}

cudaError_t kv_project_append(const KvProjArgs &a, void *ws, cudaStream_t st) {
    if (a.dt == YOCO_BF16) return run<bf16_t>(a, ws, st);
    return run<float>(a, ws, st);
}

}  // namespace yoco_host

YOCO_DEBUG_TU(kv_proj)
