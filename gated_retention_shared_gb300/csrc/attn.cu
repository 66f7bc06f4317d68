// attn.cu -- cross-decoder attention over the shared K^/V^ cache (paper Section 2.2,
// Eq. 3): causal grouped-query softmax attention, split over the key axis
// (flash-decoding) and merged by log-sum-exp.
//
// One CTA = one kv head of one sequence, a block of query rows (all query heads of
// that kv head's group, so each K/V byte is read once for the whole group) and one
// slice of the keys.  Four warps take 32 keys each of every 128-key tile: lane =
// key for the scores, lane = 4 head-dim lanes for the value sum; each warp keeps
// its own running max / sum / accumulator and the warps are merged at the end.
// K/V tiles are double-buffered in shared memory with cp.async.
#include <type_traits>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "rope.cuh"

namespace yoco {

constexpr int kAttnWarps = 4;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kAttnTile = 32 * kAttnWarps;  // keys per tile
constexpr int kAttnMaxQ = 16;               // query vectors per CTA

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

template <typename T, int D, int NQ = kAttnMaxQ> struct AttnCfg {
    static constexpr int kRowBytes = D * (int)sizeof(T);
    static constexpr int kKPitch = kRowBytes + 16;  // padded K rows: lanes read different rows
    static constexpr int kVPitch = kRowBytes;
    static constexpr int kStages = 1;  // overlap comes from 3 resident CTAs per SM
    static constexpr int kStageBytes = kAttnTile * (kKPitch + kVPitch);
    static constexpr int kEpt = D / 32;  // head-dim elements per lane
    __host__ __device__ static constexpr size_t smem_bytes() {
        size_t tiles = (size_t)kStages * kStageBytes;
        size_t merge = (size_t)kAttnWarps * NQ * (D + 2) * sizeof(float);
        return (tiles > merge ? tiles : merge) + (size_t)NQ * D * sizeof(float);
    }
};

// grid: x = key split, y = query row block, z = b * Hkv + kv head
// rows: t in [y * RB, min(T, (y + 1) * RB)); query vector qv = (t - t0) * G + g
template <typename T, int D, int NQ>
__global__ void __launch_bounds__(kAttnThreads, 3)
attn_split_kernel(const T *__restrict__ Q, T *__restrict__ O, const T *__restrict__ Kc,
                  const T *__restrict__ Vc, float *__restrict__ part, int T_rows, int Hq, int Hkv,
                  int64_t cap, int64_t p0, float scale, int RB, int64_t keys_per_split, int splits,
                  float rope_base, const RopeFreq rf) {
    using Cfg = AttnCfg<T, D, NQ>;
    constexpr int E = Cfg::kEpt;
    extern __shared__ float4 smem4[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(smem4);
    float *qs = reinterpret_cast<float *>(smem + (Cfg::smem_bytes() - (size_t)NQ * D * sizeof(float)));

    const int G = Hq / Hkv;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int split = blockIdx.x;
    const int t0 = blockIdx.y * RB;
    const int t1 = min(T_rows, t0 + RB);
    const int bz = blockIdx.z;
    const int b = bz / Hkv, hk = bz % Hkv;
    const int nq = (t1 - t0) * G;

    // queries (pre-scaled) as fp32 in shared memory
    for (int e = threadIdx.x; e < nq * D; e += kAttnThreads) {
        int qv = e / D, c = e % D;
        int t = t0 + qv / G, h = hk * G + qv % G;
        qs[e] = scale * to_f32(Q[(((size_t)b * T_rows + t) * Hq + h) * D + c]);
    }
    if (rope_base > 0.f) {  // rotary encoding: turn each query row by its position
        __syncthreads();
        for (int e = threadIdx.x; e < nq * (D / 2); e += kAttnThreads) {
            const int qv = e / (D / 2), i = e % (D / 2);
            float c, s;
            rope_cs_exact(p0 + t0 + qv / G, rf.theta[i], c, s);
            rope_turn(qs[qv * D + 2 * i], qs[qv * D + 2 * i + 1], c, s);
        }
        __syncthreads();
    }

    const int64_t k_lo = (int64_t)split * keys_per_split;
    const int64_t k_hi = min(k_lo + keys_per_split, p0 + (int64_t)t1);  // last row reads up to p0+t1-1
    if (!YOCO_DCHECK(k_lo >= 0 && p0 + (int64_t)t1 <= cap && b < (int)(gridDim.z / Hkv), 0x52)) return;
    const T *Kb = Kc + ((size_t)b * Hkv + hk) * (size_t)cap * D;
    const T *Vb = Vc + ((size_t)b * Hkv + hk) * (size_t)cap * D;

    float m[NQ], l[NQ], acc[NQ][E];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[i][e] = 0.f;
    }

    auto issue_tile = [&](int64_t base, int stage) {
        unsigned char *sk = smem + (size_t)stage * Cfg::kStageBytes;
        unsigned char *sv = sk + kAttnTile * Cfg::kKPitch;
        constexpr int chunks_per_row = Cfg::kRowBytes / 16;
        for (int e = threadIdx.x; e < kAttnTile * chunks_per_row; e += kAttnThreads) {
            int r = e / chunks_per_row, c = e % chunks_per_row;
            int64_t key = base + r;
            if (key < k_hi) {
                cp_async16(sk + r * Cfg::kKPitch + c * 16, reinterpret_cast<const unsigned char *>(Kb + key * D) + c * 16);
                cp_async16(sv + r * Cfg::kVPitch + c * 16, reinterpret_cast<const unsigned char *>(Vb + key * D) + c * 16);
            }
        }
        cp_async_commit();
    };

    __syncthreads();
    const int ntiles = (k_hi > k_lo) ? (int)((k_hi - k_lo + kAttnTile - 1) / kAttnTile) : 0;
    if (ntiles > 0) issue_tile(k_lo, 0);
    for (int it = 0; it < ntiles; ++it) {
        const int stage = (Cfg::kStages == 2) ? (it & 1) : 0;
        if constexpr (Cfg::kStages == 2) {
            if (it + 1 < ntiles) {
                issue_tile(k_lo + (int64_t)(it + 1) * kAttnTile, (it + 1) & 1);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
        } else {
            if (it > 0) issue_tile(k_lo + (int64_t)it * kAttnTile, 0);
            cp_async_wait<0>();
        }
        __syncthreads();
        const unsigned char *sk = smem + (size_t)stage * Cfg::kStageBytes;
        const unsigned char *sv = sk + kAttnTile * Cfg::kKPitch;
        const int64_t base = k_lo + (int64_t)it * kAttnTile;
        const int r = warp * 32 + lane;  // this lane's key within the tile
        const int64_t key = base + r;
        const bool key_ok = key < k_hi;

        // scores s[qv] = q_qv . k_key (q already scaled)
        float s[NQ];
#pragma unroll
        for (int i = 0; i < NQ; ++i) s[i] = 0.f;
        const T *krow = reinterpret_cast<const T *>(sk + r * Cfg::kKPitch);
        for (int c = 0; c < D; c += 4) {
            float kv[4];
            if constexpr (sizeof(T) == 2) {
                uint2 u = *reinterpret_cast<const uint2 *>(krow + c);
                kv[0] = __uint_as_float(u.x << 16);
                kv[1] = __uint_as_float(u.x & 0xFFFF0000u);
                kv[2] = __uint_as_float(u.y << 16);
                kv[3] = __uint_as_float(u.y & 0xFFFF0000u);
            } else {
                float4 f = *reinterpret_cast<const float4 *>(krow + c);
                kv[0] = f.x; kv[1] = f.y; kv[2] = f.z; kv[3] = f.w;
            }
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
                if (i < nq) {
                    float4 qq = *reinterpret_cast<const float4 *>(&qs[i * D + c]);
                    s[i] = fmaf(qq.x, kv[0], fmaf(qq.y, kv[1], fmaf(qq.z, kv[2], fmaf(qq.w, kv[3], s[i]))));
                }
            }
        }
        // causal mask + online softmax per query vector (warp-wide over its 32 keys)
        const T *vbase = reinterpret_cast<const T *>(sv);
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            if (i >= nq) break;
            const int64_t pos = p0 + t0 + i / G;
            float si = (key_ok && key <= pos) ? s[i] : -INFINITY;
            float mx = si;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_new = fmaxf(m[i], mx);
            float pexp = (m_new == -INFINITY) ? 0.f : __expf(si - m_new);
            const float corr = (m_new == -INFINITY) ? 1.f : __expf(m[i] - m_new);
            float psum = pexp;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
            l[i] = l[i] * corr + psum;
            m[i] = m_new;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[i][e] *= corr;
            s[i] = pexp;
        }
        // acc[qv][lane dims] += sum_j p_j v_j over this warp's valid keys (rows past
        // k_hi were never loaded and may hold anything)
        const int64_t warp_first = base + warp * 32;
        const int nvalid = (int)max((int64_t)0, min((int64_t)32, k_hi - warp_first));
        for (int j = 0; j < nvalid; ++j) {
            const int rj = warp * 32 + j;
            float vv[E];
            const T *vrow = vbase + (size_t)rj * (Cfg::kVPitch / sizeof(T)) + lane * E;
            if constexpr (sizeof(T) == 2 && E == 4) {
                uint2 u = *reinterpret_cast<const uint2 *>(vrow);
                vv[0] = __uint_as_float(u.x << 16);
                vv[1] = __uint_as_float(u.x & 0xFFFF0000u);
                vv[2] = __uint_as_float(u.y << 16);
                vv[3] = __uint_as_float(u.y & 0xFFFF0000u);
            } else if constexpr (sizeof(T) == 2) {
                uint32_t u = *reinterpret_cast<const uint32_t *>(vrow);
                vv[0] = __uint_as_float(u << 16);
                vv[1] = __uint_as_float(u & 0xFFFF0000u);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) vv[e] = vrow[e];
            }
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
                if (i < nq) {
                    float pj = __shfl_sync(0xffffffffu, s[i], j);
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[i][e] = fmaf(pj, vv[e], acc[i][e]);
                }
            }
        }
        __syncthreads();  // stage is reused by the next issue
    }

    // merge the four warps
    float *mw = reinterpret_cast<float *>(smem);              // [warps][MaxQ][D + 2]
    const int pitch = D + 2;
    for (int i = 0; i < nq; ++i) {
        float *row = mw + ((size_t)warp * NQ + i) * pitch;
#pragma unroll
        for (int e = 0; e < E; ++e) row[lane * E + e] = acc[i][e];
        if (lane == 0) {
            row[D] = m[i];
            row[D + 1] = l[i];
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < nq * D; e += kAttnThreads) {
        const int i = e / D, c = e % D;
        float M = -INFINITY;
        for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, mw[((size_t)w * NQ + i) * pitch + D]);
        float L = 0.f, A = 0.f;
        for (int w = 0; w < kAttnWarps; ++w) {
            const float *row = mw + ((size_t)w * NQ + i) * pitch;
            float f = (row[D] == -INFINITY) ? 0.f : __expf(row[D] - M);
            L += row[D + 1] * f;
            A += row[c] * f;
        }
        const int t = t0 + i / G, h = hk * G + i % G;
        const size_t qrow = ((size_t)b * T_rows + t) * Hq + h;
        if (!YOCO_DCHECK(t < T_rows && h < Hq && split < splits, 0x53)) continue;
        if (splits == 1) {
            O[qrow * D + c] = from_f32<T>(A / L);
        } else {
            float *pp = part + (qrow * splits + split) * (D + 2);
            pp[c] = A;
            if (c == 0) {
                pp[D] = M;
                pp[D + 1] = L;
            }
        }
    }
}

// merge the splits of every query row by log-sum-exp: one CTA per (row, head),
// thread c owns head dim c.  Splits are taken kCombineBatch at a time; every
// thread issues all of a batch's loads at once (each split's maximum and sum,
// the same addresses across the CTA, and its own column of the partial
// outputs), so a batch costs one L2 round trip, and the batches are folded
// online (running maximum, rescaled sum and output).  Partials are read past
// L1 (the split kernel wrote them from other SMs).
constexpr int kCombineMaxSplits = 4096;
constexpr int kCombineBatch = 32;

template <typename T, int D>
__global__ void __launch_bounds__(D) attn_combine_kernel(const float *__restrict__ part, T *__restrict__ O, int splits) {
    // launched as a programmatic dependent of the split kernel: wait for its partials
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    const int w = blockIdx.x, c = threadIdx.x;
    const float *pp = part + (size_t)w * splits * (D + 2);
    float M = -INFINITY, L = 0.f, A = 0.f;
    for (int s0 = 0; s0 < splits; s0 += kCombineBatch) {
        const int n = min(kCombineBatch, splits - s0);
        float ms[kCombineBatch], ls[kCombineBatch], os[kCombineBatch];
#pragma unroll
        for (int j = 0; j < kCombineBatch; ++j) {
            if (j < n) {
                const float *q = pp + (size_t)(s0 + j) * (D + 2);
                ms[j] = __ldcg(q + D);
                ls[j] = __ldcg(q + D + 1);
                os[j] = __ldcg(q + c);
            } else {
                ms[j] = -INFINITY;
                ls[j] = 0.f;
                os[j] = 0.f;
            }
        }
        float mb = M;
#pragma unroll
        for (int j = 0; j < kCombineBatch; ++j) mb = fmaxf(mb, ms[j]);
        if (mb == -INFINITY) continue;  // nothing valid so far
        const float r = (M == -INFINITY) ? 0.f : __expf(M - mb);
        L *= r;
        A *= r;
#pragma unroll
        for (int j = 0; j < kCombineBatch; ++j) {
            const float f = (ms[j] == -INFINITY) ? 0.f : __expf(ms[j] - mb);
            L = fmaf(ls[j], f, L);
            A = fmaf(os[j], f, A);
        }
        M = mb;
    }
    if (YOCO_DCHECK(w < (int)gridDim.x, 0x54)) O[(size_t)w * D + c] = from_f32<T>(A / L);
}

}  // namespace yoco

namespace yoco_host {
using namespace yoco;

constexpr int kFaMinRows = 64;  // from this many query rows on, prefill uses attn_fa_kernel

static int rows_per_block(int G) { return G >= kAttnMaxQ ? 1 : kAttnMaxQ / G; }

int attn_auto_splits(int B, int Hkv, int64_t keys, int ctas_per_sm) {
    // Split count for B*Hkv (sequence, kv head) units: at least one full wave of
    // CTAs on the device's SMs, then the smallest count whose last wave is >= 95 % full
    // (on 152 SMs: 8 units take 19 splits = 152 CTAs, 64 units 7 = 448 of 456 slots,
    // 256 units 4 = 1024 of 1064), never more than one split per two key tiles.
    const int64_t units = (int64_t)B * Hkv;
    const int64_t slots = (int64_t)ctas_per_sm * device_sm_count();
    int64_t cap = (keys + 2 * kAttnTile - 1) / (2 * kAttnTile);
    if (cap > 1024) cap = 1024;
    if (cap < 1) cap = 1;
    int64_t s_min = (slots + units - 1) / units;
    if (s_min > cap) s_min = cap;
    const int64_t s_max = std::min<int64_t>(cap, 8 * s_min);
    int64_t best = s_min;
    double best_eff = -1.0;
    for (int64_t s = s_min; s <= s_max; ++s) {
        const int64_t ctas = units * s;
        const double eff = (double)ctas / (double)(slots * ((ctas + slots - 1) / slots));
        if (eff >= 0.95) return (int)s;
        if (eff > best_eff) {
            best_eff = eff;
            best = s;
        }
    }
    return (int)best;
}

// workspace: [0, 256) status word of the tensor-core kernel, then the split partials
int attn_ctas_per_sm(yoco_dtype dt, int d, int group) { return (dt == YOCO_BF16 && d == 128 && group <= 16) ? 1 : 3; }

size_t attn_workspace(int B, int Hq, int T, int d, int splits) {
    if (splits <= 1) return 256;
    return 256 + (size_t)B * T * Hq * splits * (d + 2) * sizeof(float);
}

template <typename T, int D, int NQ>
static cudaError_t launch_nq(const AttnArgs &a, int RB, int64_t kps, int splits, void *ws, cudaStream_t st) {
    auto kern = attn_split_kernel<T, D, NQ>;
    size_t smem = AttnCfg<T, D, NQ>::smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(splits, (a.T + RB - 1) / RB, a.B * a.Hkv);
    count_launches(splits > 1 ? 2 : 1);
    kern<<<grid, kAttnThreads, smem, st>>>((const T *)a.Q, (T *)a.O, (const T *)a.kc, (const T *)a.vc, (float *)ws,
                                           a.T, a.Hq, a.Hkv, a.cap, a.p0, a.scale, RB, kps, splits, a.rope_base, make_rope_freq(a.rope_base, D));
    return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t launch(const AttnArgs &a, int splits, void *ws, cudaStream_t st) {
    const int G = a.Hq / a.Hkv;
    const int RB = rows_per_block(G);
    const int64_t keys = a.p0 + a.T;  // positions 0 .. p0+T-1
    int64_t kps = (keys + splits - 1) / splits;
    kps = ((kps + kAttnTile - 1) / kAttnTile) * kAttnTile;
    splits = (int)((keys + kps - 1) / kps);
    if (splits > kCombineMaxSplits) return cudaErrorInvalidValue;  // the merge holds one factor per split
    const int nq = (a.T < RB ? a.T : RB) * G;  // query vectors per CTA
    const int rb_eff = (nq <= 4 && a.T <= RB) ? a.T : RB;
    float *part = (float *)((char *)ws + 256);
    cudaError_t e;
    // many rows (prefill): 128-row query tiles on the tensor cores, no key splits
    if (std::is_same<T, bf16_t>::value && a.T >= kFaMinRows && attn_fa_eligible(a))
        return attn_fa_launch(a, 0, (int *)ws, st);
    if (std::is_same<T, bf16_t>::value && attn_tc_eligible(a, nq)) {
        count_launches(splits > 1 ? 2 : 1);
        e = attn_tc_launch(a, rb_eff, nq, kps, splits, part, (int *)ws, st);
    } else if (nq <= 4) e = launch_nq<T, D, 4>(a, rb_eff, kps, splits, part, st);
    else if (nq <= 8) e = launch_nq<T, D, 8>(a, RB, kps, splits, part, st);
    else e = launch_nq<T, D, 16>(a, RB, kps, splits, part, st);
    if (e != cudaSuccess) return e;
    if (splits > 1) {
        const int rows = a.B * a.T * a.Hq;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(rows);
        cfg.blockDim = dim3(D);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, attn_combine_kernel<T, D>, (const float *)part, (T *)a.O, splits);
    }
    return e;
}

cudaError_t attn_run(const AttnArgs &a, int splits, void *ws, cudaStream_t st) {
    if (a.dt == YOCO_BF16) {
        if (a.d == 64) return launch<bf16_t, 64>(a, splits, ws, st);
        return launch<bf16_t, 128>(a, splits, ws, st);
    }
    if (a.d == 64) return launch<float, 64>(a, splits, ws, st);
    return launch<float, 128>(a, splits, ws, st);
}

}  // namespace yoco_host

YOCO_DEBUG_TU(attn)
