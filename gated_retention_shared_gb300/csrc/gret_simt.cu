// gret_simt.cu -- gated retention on CUDA cores (fp32 FMA).
//
//  * gret_chunk_simt: the chunkwise form (paper Section 3.1, Eq. 6 with the row
//    convention made consistent; Appendix F ChunkwiseRetention) for one
//    (sequence, head, 64-column slice of d_v, segment of the sequence).  In
//    WRITE_O mode it writes o and the segment's end state from a given initial
//    state; in state-only mode it returns the segment's end state from a zero
//    initial state plus the segment's total log decay.
//  * gret_segment_scan: joins segment end states into each segment's initial
//    state, S_start(p+1) = exp(G_p) S_start(p) + E_p, and the final state.
//  * gret_decode_step: the recurrent form for one token (Eq. 5).
//
// Used for fp32 inputs, for head sizes or shapes the tensor-core kernel does not
// take, and as the sequence-parallel scan shared with the tensor-core path.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace yoco {

constexpr int kSimtC = 64;    // chunk length
constexpr int kSimtDVB = 64;  // d_v columns per CTA
constexpr int kSimtThreads = 256;
constexpr int kPad = 4;  // row padding (floats) of the transposed tiles

__host__ __device__ constexpr size_t simt_smem_floats(int DK) {
    return (size_t)DK * (kSimtC + kPad) * 2   // Qt, Kt  [DK][C+pad]
           + (size_t)kSimtC * DK              // Kw      [C][DK]
           + (size_t)kSimtC * kSimtDVB        // Vs      [C][DVB]
           + (size_t)kSimtC * (kSimtC + kPad) // Pt      [C][C+pad]
           + (size_t)DK * kSimtDVB            // S       [DK][DVB]
           + kSimtC;                          // b       [C]
}

// grid: x = segment * (dv / 64) + dv block, y = head, z = sequence.
// Segment p covers tokens [p * seg_len, min(N, (p + 1) * seg_len)), seg_len % 64 == 0.
// S_in / S_out / G_out index (b, h, p) as ((b * H + h) * P + p); S_in may be null (zeros).
template <typename Tin, typename Tout, int DK, bool WRITE_O>
__global__ void __launch_bounds__(kSimtThreads)
gret_chunk_simt(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                const float *__restrict__ logits, float inv_tau, Tout *__restrict__ o,
                const float *__restrict__ S_in, float *__restrict__ S_out, float *__restrict__ G_out,
                int N, int H, int dv, int seg_len, int P) {
    constexpr int C = kSimtC, DVB = kSimtDVB, LDT = kSimtC + kPad;
    constexpr int RS = DK / 16;  // state rows per thread in the update
    extern __shared__ float4 smem4[];
    float *smem = reinterpret_cast<float *>(smem4);
    float *Qt = smem;
    float *Kt = Qt + DK * LDT;
    float *Kw = Kt + DK * LDT;
    float *Vs = Kw + C * DK;
    float *Pt = Vs + C * DVB;
    float *S = Pt + C * LDT;
    float *bsh = S + DK * DVB;

    const int tid = threadIdx.x;
    const int ndvb = dv / DVB;
    const int p = blockIdx.x / ndvb;
    const int dv0 = (blockIdx.x % ndvb) * DVB;
    const int h = blockIdx.y, b = blockIdx.z;
    const int t_begin = p * seg_len;
    const int t_end = min(N, t_begin + seg_len);
    const size_t bhp = ((size_t)b * H + h) * P + p;
    const size_t row_stride_k = (size_t)H * DK, row_stride_v = (size_t)H * dv;

    // state slice S[:, dv0:dv0+64]
    for (int e = tid; e < DK * DVB; e += kSimtThreads) {
        int i = e / DVB, c = e % DVB;
        S[e] = S_in ? S_in[bhp * DK * dv + (size_t)i * dv + dv0 + c] : 0.0f;
    }
    float seg_decay = 0.0f;  // sum of log gates over the segment
    __syncthreads();

    for (int c0 = t_begin; c0 < t_end; c0 += C) {
        const int len = min(C, t_end - c0);
        if (tid < C) {
            float lg = 0.0f;
            if (tid < len) lg = log_gate(logits[((size_t)b * N + c0 + tid) * H + h], inv_tau);
            bsh[tid] = lg;
        }
        __syncthreads();
        if (tid == 0) {  // chunk-local cumulative log decay b_j (padding rows add 0)
            float acc = 0.0f;
            for (int j = 0; j < C; ++j) {
                acc += bsh[j];
                bsh[j] = acc;
            }
        }
        __syncthreads();
        const float bC = bsh[C - 1];
        seg_decay += bC;
        for (int e = tid; e < C * DK; e += kSimtThreads) {
            int j = e / DK, i = e % DK;
            float qv = 0.0f, kv = 0.0f;
            if (j < len) {
                size_t base = (((size_t)b * N + c0 + j) * H + h) * DK + i;
                qv = to_f32(q[base]);
                kv = to_f32(k[base]);
            }
            Qt[i * LDT + j] = qv;
            Kt[i * LDT + j] = kv;
            Kw[j * DK + i] = kv * expf(bC - bsh[j]);  // decay of token j to the chunk end
        }
        for (int e = tid; e < C * DVB; e += kSimtThreads) {
            int j = e / DVB, c = e % DVB;
            Vs[e] = (j < len) ? to_f32(v[(((size_t)b * N + c0 + j) * H + h) * dv + dv0 + c]) : 0.0f;
        }
        (void)row_stride_k;
        (void)row_stride_v;
        __syncthreads();

        if constexpr (WRITE_O) {
            // intra-chunk scores (Q K^T) masked by D_jk = exp(b_j - b_k) [k <= j]
            {
                const int jb = tid / 16, kb = tid % 16;
                float acc[4][4] = {};
                for (int i = 0; i < DK; ++i) {
                    float4 qa = *reinterpret_cast<const float4 *>(&Qt[i * LDT + 4 * jb]);
                    float4 ka = *reinterpret_cast<const float4 *>(&Kt[i * LDT + 4 * kb]);
                    float qr[4] = {qa.x, qa.y, qa.z, qa.w}, kr[4] = {ka.x, ka.y, ka.z, ka.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int s = 0; s < 4; ++s) acc[r][s] = fmaf(qr[r], kr[s], acc[r][s]);
                }
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        int j = 4 * jb + r, kk = 4 * kb + s;
                        Pt[kk * LDT + j] = (kk <= j) ? acc[r][s] * expf(bsh[j] - bsh[kk]) : 0.0f;
                    }
            }
            __syncthreads();
            // o_j = sum_k P_jk v_k + exp(b_j) q_j S
            {
                const int jb = tid / 16, cb = tid % 16;
                float oa[4][4] = {}, xa[4][4] = {};
                for (int kk = 0; kk < C; ++kk) {
                    float4 pa = *reinterpret_cast<const float4 *>(&Pt[kk * LDT + 4 * jb]);
                    float4 va = *reinterpret_cast<const float4 *>(&Vs[kk * DVB + 4 * cb]);
                    float pr[4] = {pa.x, pa.y, pa.z, pa.w}, vr[4] = {va.x, va.y, va.z, va.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int s = 0; s < 4; ++s) oa[r][s] = fmaf(pr[r], vr[s], oa[r][s]);
                }
                for (int i = 0; i < DK; ++i) {
                    float4 qa = *reinterpret_cast<const float4 *>(&Qt[i * LDT + 4 * jb]);
                    float4 sa = *reinterpret_cast<const float4 *>(&S[i * DVB + 4 * cb]);
                    float qr[4] = {qa.x, qa.y, qa.z, qa.w}, sr[4] = {sa.x, sa.y, sa.z, sa.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int s = 0; s < 4; ++s) xa[r][s] = fmaf(qr[r], sr[s], xa[r][s]);
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    int j = 4 * jb + r;
                    if (j < len) {
                        float eb = expf(bsh[j]);
                        Tout *orow = o + (((size_t)b * N + c0 + j) * H + h) * dv + dv0 + 4 * cb;
#pragma unroll
                        for (int s = 0; s < 4; ++s) orow[s] = from_f32<Tout>(oa[r][s] + eb * xa[r][s]);
                    }
                }
            }
            __syncthreads();  // every read of S is done before the update
        }

        // S <- exp(b_C) S + sum_k exp(b_C - b_k) k_k^T v_k
        {
            const int ib = tid / 16, cb = tid % 16;
            const float ebC = expf(bC);
            float sa[RS][4];
#pragma unroll
            for (int r = 0; r < RS; ++r) {
                float4 s4 = *reinterpret_cast<const float4 *>(&S[(RS * ib + r) * DVB + 4 * cb]);
                sa[r][0] = s4.x * ebC;
                sa[r][1] = s4.y * ebC;
                sa[r][2] = s4.z * ebC;
                sa[r][3] = s4.w * ebC;
            }
            for (int kk = 0; kk < C; ++kk) {
                float4 va = *reinterpret_cast<const float4 *>(&Vs[kk * DVB + 4 * cb]);
                float vr[4] = {va.x, va.y, va.z, va.w};
#pragma unroll
                for (int r = 0; r < RS; ++r) {
                    float kw = Kw[kk * DK + RS * ib + r];
#pragma unroll
                    for (int s = 0; s < 4; ++s) sa[r][s] = fmaf(kw, vr[s], sa[r][s]);
                }
            }
            __syncthreads();
#pragma unroll
            for (int r = 0; r < RS; ++r)
                *reinterpret_cast<float4 *>(&S[(RS * ib + r) * DVB + 4 * cb]) =
                    make_float4(sa[r][0], sa[r][1], sa[r][2], sa[r][3]);
        }
        __syncthreads();
    }

    if (S_out) {
        for (int e = tid; e < DK * DVB; e += kSimtThreads) {
            int i = e / DVB, c = e % DVB;
            S_out[bhp * DK * dv + (size_t)i * dv + dv0 + c] = S[e];
        }
    }
    if (G_out && tid == 0 && (blockIdx.x % ndvb) == 0) G_out[bhp] = seg_decay;
}

// Sequential join of P segment states for every (b, h); parallel over the d_k x d_v
// entries.  In place: on entry E[p] holds segment p's zero-start end state, on exit
// it holds segment p's true initial state.  `state` holds the initial state on entry
// and the final state on exit.  grid: x = entry blocks, y = b * H + h.
__global__ void gret_segment_scan(float *__restrict__ E, const float *__restrict__ G,
                                  float *__restrict__ state, int P, int DD) {
    const int bh = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= DD) return;
    float s = state[(size_t)bh * DD + e];
    for (int p = 0; p < P; ++p) {
        size_t idx = ((size_t)bh * P + p) * DD + e;
        float loc = E[idx];
        E[idx] = s;
        s = expf(G[(size_t)bh * P + p]) * s + loc;
    }
    state[(size_t)bh * DD + e] = s;
}

// One recurrent step S <- gamma S + k^T v, o = q S for one (b, h) and a 32-column
// slice of d_v.  256 threads: 8 columns groups of 4 (float4) x 32 row groups.
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256)
gret_decode_step_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                        const float *__restrict__ logits, float inv_tau, float *__restrict__ state,
                        Tout *__restrict__ o, int H, int dk, int dv) {
    __shared__ float qs[128], ks[128], vs[32];
    __shared__ float part[32][33];
    const int bh = blockIdx.y;
    const int c0 = blockIdx.x * 32;
    const int tid = threadIdx.x;
    const int cg = tid % 8;   // columns c0 + 4 cg .. +3
    const int rg = tid / 8;   // rows rg, rg + 32, ...
    (void)YOCO_DCHECK(c0 + 32 <= dv && dk <= 128 && bh < (int)gridDim.y, 0x58);
    // launched as a programmatic dependent of the previous kernel on the stream: let
    // the next one start its launch, then wait for this one's inputs
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    // this thread's state rows first (dk <= 128: at most 4 rows), so their loads
    // and those of q, k, v are in flight together
    float *Sb = state + (size_t)bh * dk * dv;
    float4 srow[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = rg + 32 * u;
        if (i < dk) srow[u] = *reinterpret_cast<const float4 *>(Sb + (size_t)i * dv + c0 + 4 * cg);
    }
    for (int i = tid; i < dk; i += 256) {
        qs[i] = to_f32(q[(size_t)bh * dk + i]);
        ks[i] = to_f32(k[(size_t)bh * dk + i]);
    }
    if (tid < 32) vs[tid] = to_f32(v[(size_t)bh * dv + c0 + tid]);
    const float gamma = expf(log_gate(logits[bh], inv_tau));
    __syncthreads();
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = rg + 32 * u;
        if (i >= dk) break;
        float4 s = srow[u];
        const float ki = ks[i], qi = qs[i];
        s.x = fmaf(gamma, s.x, ki * vs[4 * cg + 0]);
        s.y = fmaf(gamma, s.y, ki * vs[4 * cg + 1]);
        s.z = fmaf(gamma, s.z, ki * vs[4 * cg + 2]);
        s.w = fmaf(gamma, s.w, ki * vs[4 * cg + 3]);
        *reinterpret_cast<float4 *>(Sb + (size_t)i * dv + c0 + 4 * cg) = s;
        acc[0] = fmaf(qi, s.x, acc[0]);
        acc[1] = fmaf(qi, s.y, acc[1]);
        acc[2] = fmaf(qi, s.z, acc[2]);
        acc[3] = fmaf(qi, s.w, acc[3]);
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) part[rg][4 * cg + s] = acc[s];
    __syncthreads();
    if (tid < 32) {
        float sum = 0.f;
        for (int r = 0; r < 32; ++r) sum += part[r][tid];
        o[(size_t)bh * dv + c0 + tid] = from_f32<Tout>(sum);
    }
}


// The recurrent step followed by the output of multi-head gated retention (paper
// Section 3.1, Eq. 7): z = swish(gate) (.) GroupNorm_h(o), one group per head.  The
// dv/32 CTAs of one head form a cluster: each computes its 32 columns of o as the
// plain step does, pushes the sum and the sum of squares of its columns into every
// peer's shared memory, passes one cluster barrier, and normalises and gates its
// own columns from the head totals (variance E[o^2] - E[o]^2, biased, in fp32).
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256)
gret_decode_step_gn_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                           const float *__restrict__ logits, float inv_tau, float *__restrict__ state,
                           const Tin *__restrict__ gate, const float *__restrict__ gn_w,
                           const float *__restrict__ gn_b, float eps, Tout *__restrict__ z, int H, int dk, int dv) {
    __shared__ float qs[128], ks[128], vs[32];
    __shared__ float part[32][33];
    __shared__ __align__(8) float red[4][2];  // (sum, sum of squares) of each CTA of the cluster, by rank
    const int bh = blockIdx.y;
    const int c0 = blockIdx.x * 32;
    const int tid = threadIdx.x;
    const int cg = tid % 8;
    const int rg = tid / 8;
    const uint32_t rank = tc::cluster_ctarank();
    const uint32_t nrank = (uint32_t)(dv / 32);
    (void)YOCO_DCHECK(c0 + 32 <= dv && dk <= 128, 0x58);
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    float *Sb = state + (size_t)bh * dk * dv;
    float4 srow[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = rg + 32 * u;
        if (i < dk) srow[u] = *reinterpret_cast<const float4 *>(Sb + (size_t)i * dv + c0 + 4 * cg);
    }
    for (int i = tid; i < dk; i += 256) {
        qs[i] = to_f32(q[(size_t)bh * dk + i]);
        ks[i] = to_f32(k[(size_t)bh * dk + i]);
    }
    if (tid < 32) vs[tid] = to_f32(v[(size_t)bh * dv + c0 + tid]);
    const float g_in = (tid < 32) ? to_f32(gate[(size_t)bh * dv + c0 + tid]) : 0.f;
    const float gamma = expf(log_gate(logits[bh], inv_tau));
    __syncthreads();
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = rg + 32 * u;
        if (i >= dk) break;
        float4 s = srow[u];
        const float ki = ks[i], qi = qs[i];
        s.x = fmaf(gamma, s.x, ki * vs[4 * cg + 0]);
        s.y = fmaf(gamma, s.y, ki * vs[4 * cg + 1]);
        s.z = fmaf(gamma, s.z, ki * vs[4 * cg + 2]);
        s.w = fmaf(gamma, s.w, ki * vs[4 * cg + 3]);
        *reinterpret_cast<float4 *>(Sb + (size_t)i * dv + c0 + 4 * cg) = s;
        acc[0] = fmaf(qi, s.x, acc[0]);
        acc[1] = fmaf(qi, s.y, acc[1]);
        acc[2] = fmaf(qi, s.z, acc[2]);
        acc[3] = fmaf(qi, s.w, acc[3]);
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) part[rg][4 * cg + s] = acc[s];
    __syncthreads();
    if (tid < 32) {
        float ov = 0.f;
        for (int r = 0; r < 32; ++r) ov += part[r][tid];
        float s1 = ov, s2 = ov * ov;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            s1 += __shfl_xor_sync(0xffffffffu, s1, off);
            s2 += __shfl_xor_sync(0xffffffffu, s2, off);
        }
        if (tid < (int)nrank) {  // lane p writes this CTA's sums into CTA p's table
            const uint32_t dst = tc::mapa_shared(&red[rank][0], (uint32_t)tid);
            asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};\n" ::"r"(dst), "f"(s1), "f"(s2) : "memory");
        }
        part[0][tid] = ov;  // kept for the normalisation below (row 0 is read above only by this thread)
    }
    tc::cluster_sync();  // every CTA's sums are in every CTA's table
    if (tid < 32) {
        float t1 = 0.f, t2 = 0.f;
        for (uint32_t r = 0; r < nrank; ++r) {
            t1 += red[r][0];
            t2 += red[r][1];
        }
        const float mean = t1 / (float)dv;
        const float var = fmaxf(t2 / (float)dv - mean * mean, 0.f);
        const float inv = rsqrtf(var + eps);
        const int h = bh % H, c = c0 + tid;
        float y = (part[0][tid] - mean) * inv;
        if (gn_w) y *= gn_w[(size_t)h * dv + c];
        if (gn_b) y += gn_b[(size_t)h * dv + c];
        const float sw = g_in / (1.f + __expf(-g_in));  // swish(g) = g sigmoid(g)
        z[(size_t)bh * dv + c] = from_f32<Tout>(sw * y);
    }
}

}  // namespace yoco

// ------------------------------------------------------------------ host side
namespace yoco_host {

using namespace yoco;

size_t gret_simt_smem_bytes(int dk) { return simt_smem_floats(dk) * sizeof(float); }

template <typename Tin, typename Tout, int DK, bool WO>
static cudaError_t launch_chunk(const GretArgs &a, const float *S_in, float *S_out, float *G_out,
                                int seg_len, int P, cudaStream_t st) {
    auto kern = gret_chunk_simt<Tin, Tout, DK, WO>;
    size_t smem = simt_smem_floats(DK) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(P * (a.dv / kSimtDVB), a.H, a.B);
    count_launches(1);
    kern<<<grid, kSimtThreads, smem, st>>>((const Tin *)a.q, (const Tin *)a.k, (const Tin *)a.v, a.logits,
                                           1.0f / a.tau, (Tout *)a.o, S_in, S_out, G_out, a.N, a.H, a.dv,
                                           seg_len, P);
    return cudaGetLastError();
}

template <typename Tin, typename Tout, int DK>
static cudaError_t run_simt(const GretArgs &a, int P, int seg_len, float *ws, cudaStream_t st) {
    cudaError_t e;
    if (P == 1) return launch_chunk<Tin, Tout, DK, true>(a, a.state, a.state, nullptr, seg_len, 1, st);
    const size_t DD = (size_t)a.dk * a.dv;
    float *E = ws;                                   // [B, H, P, dk, dv]
    float *G = ws + (size_t)a.B * a.H * P * DD;      // [B, H, P]
    e = launch_chunk<Tin, Tout, DK, false>(a, nullptr, E, G, seg_len, P, st);
    if (e != cudaSuccess) return e;
    dim3 g2((unsigned)((DD + 255) / 256), a.B * a.H);
    count_launches(1);
    gret_segment_scan<<<g2, 256, 0, st>>>(E, G, a.state, P, (int)DD);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_chunk<Tin, Tout, DK, true>(a, E, nullptr, nullptr, seg_len, P, st);
}

cudaError_t gret_scan_launch(float *E, const float *G, float *state, int BH, int P, int DD, cudaStream_t st) {
    dim3 g2((unsigned)((DD + 255) / 256), BH);
    gret_segment_scan<<<g2, 256, 0, st>>>(E, G, state, P, DD);
    return cudaGetLastError();
}

int gret_simt_segments(int B, int N, int H, int dv) {
    // enough CTAs to cover the GPU about once; each segment at least one chunk
    int ctas = B * H * (dv / kSimtDVB);
    int chunks = (N + kSimtC - 1) / kSimtC;
    const int sms = device_sm_count();
    int P = (ctas >= sms) ? 1 : (sms + ctas - 1) / ctas;
    if (P > chunks) P = chunks;
    if (P < 1) P = 1;
    return P;
}

int gret_simt_seg_len(int N, int P) {
    int chunks = (N + kSimtC - 1) / kSimtC;
    return ((chunks + P - 1) / P) * kSimtC;
}

size_t gret_simt_workspace(int B, int N, int H, int dk, int dv) {
    int P = gret_simt_segments(B, N, H, dv);
    if (P == 1) return 0;
    return ((size_t)B * H * P * dk * dv + (size_t)B * H * P) * sizeof(float);
}

cudaError_t gret_prefill_simt(const GretArgs &a, void *ws, cudaStream_t st) {
    int P = gret_simt_segments(a.B, a.N, a.H, a.dv);
    int seg_len = gret_simt_seg_len(a.N, P);
    P = (a.N + seg_len - 1) / seg_len;  // drop empty trailing segments
    if (P < 1) P = 1;
    float *w = (float *)ws;
    if (a.in_dt == YOCO_F32) {
        if (a.dk == 64) return run_simt<float, float, 64>(a, P, seg_len, w, st);
        return run_simt<float, float, 128>(a, P, seg_len, w, st);
    } else {
        if (a.dk == 64) return run_simt<bf16_t, bf16_t, 64>(a, P, seg_len, w, st);
        return run_simt<bf16_t, bf16_t, 128>(a, P, seg_len, w, st);
    }
}

cudaError_t gret_decode_gn(const void *q, const void *k, const void *v, const float *logits, float tau,
                           float *state, const void *gate, const float *gn_w, const float *gn_b, float eps, void *z,
                           int B, int H, int dk, int dv, yoco_dtype dt, cudaStream_t st) {
    // the dv/32 column slices of one head form a cluster; a programmatic dependent
    // of the previous kernel like the plain step
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(dv / 32, B * H);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = dv / 32;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    count_launches(1);
    if (dt == YOCO_F32)
        return cudaLaunchKernelEx(&cfg, gret_decode_step_gn_kernel<float, float>, (const float *)q, (const float *)k,
                                  (const float *)v, logits, 1.0f / tau, state, (const float *)gate, gn_w, gn_b, eps,
                                  (float *)z, H, dk, dv);
    return cudaLaunchKernelEx(&cfg, gret_decode_step_gn_kernel<bf16_t, bf16_t>, (const bf16_t *)q,
                              (const bf16_t *)k, (const bf16_t *)v, logits, 1.0f / tau, state, (const bf16_t *)gate,
                              gn_w, gn_b, eps, (bf16_t *)z, H, dk, dv);
}

cudaError_t gret_decode(const void *q, const void *k, const void *v, const float *logits, float tau,
                        float *state, void *o, int B, int H, int dk, int dv, yoco_dtype dt, cudaStream_t st) {
    // a programmatic dependent of the previous kernel: in a run of layers (or a
    // captured graph of them) each step's launch overlaps the previous step
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(dv / 32, B * H);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launches(1);
    if (dt == YOCO_F32)
        return cudaLaunchKernelEx(&cfg, gret_decode_step_kernel<float, float>, (const float *)q, (const float *)k,
                                  (const float *)v, logits, 1.0f / tau, state, (float *)o, H, dk, dv);
    return cudaLaunchKernelEx(&cfg, gret_decode_step_kernel<bf16_t, bf16_t>, (const bf16_t *)q, (const bf16_t *)k,
                              (const bf16_t *)v, logits, 1.0f / tau, state, (bf16_t *)o, H, dk, dv);
}

}  // namespace yoco_host

YOCO_DEBUG_TU(gret_simt)
