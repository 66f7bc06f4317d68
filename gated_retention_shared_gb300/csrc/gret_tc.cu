// gret_tc.cu -- chunkwise gated retention on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA), bf16 inputs, head size 128, 128-token chunks.
//
// Math (paper Section 3.1, Eq. 6 with consistent indices; Appendix F
// ChunkwiseRetention).  For a chunk with chunk-local cumulative log decay b_j
// (b_j = sum of log gamma over the chunk's tokens up to and including j) and the
// state S (d_k x d_v) before the chunk:
//     o_j  = sum_{k<=j} (q_j . k_k) e^{b_j - b_k} v_k  +  e^{b_j} q_j S
//     S'   = e^{b_C} S + sum_k e^{b_C - b_k} k_k^T v_k
// Everything is computed transposed, so that one TMEM lane holds one d_v column
// and the output leaves TMEM as coalesced rows:
//     A    = Q K^T                       (lane = query j)         MMA1
//     P_jk = A_jk e^{b_j - b_k} [k <= j] (bf16, shared memory)
//     O^T  = V^T P^T + S^T Q'^T,  Q'_j = e^{b_j} q_j               MMA2, MMA3
//     U^T  = V^T K',              K'_k = e^{b_C - b_k} k_k         MMA4
//     S'^T = e^{b_C} S^T + U^T   (fp32, registers of the state warps)
// S^T is fed back to MMA3 as a bf16 A operand in TMEM; the fp32 state never
// leaves the registers until the segment ends.
//
// Sequence parallelism: the sequence of every (b, h) is cut into P segments of
// whole chunks.  Kernel mode SEG_STATE walks a segment backwards and accumulates
// its zero-start end state  E^T = sum_k e^{(decay after k to segment end)} v_k^T k_k
// directly in TMEM (every weight <= 1), plus the segment's total log decay.  A
// small scan (gret_simt.cu) turns those into each segment's initial state, and
// mode OUTPUT runs the chunk recurrence above from it.  With B*H >= #SMs, P = 1
// and only OUTPUT runs.
//
// Warp roles (320 threads): warps 0-3 state + output epilogue (thread = TMEM lane
// = d_v column), warps 4-7 decay / P / in-place scaling of Q and K (thread = token
// row of the chunk), warp 8 TMA producer, warp 9 MMA issuer.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace yoco {

using namespace tc;

constexpr int kC = 128;                     // chunk length = MMA M/N
constexpr int kD = 128;                     // head size
constexpr int kTile = kC * kD * 2;          // 32 KB bf16 tile
constexpr int kHalf = kTile / 2;            // one 64-column block
constexpr int kStages = 2;
constexpr int kTcThreads = 320;

// TMEM columns
constexpr uint32_t kColA = 0, kColO = 128, kColU = 256, kColS = 384;

enum : int { MODE_OUTPUT = 0, MODE_SEG_STATE = 1 };

struct TcSmem {
    uint64_t full[kStages], empty[kStages], pq_ready[kStages];
    uint64_t as_full, as_free, o_full, o_free, u_full, u_free, s_ready, drain;
    uint32_t tmem_base;
    int abort_flag;
    int go0, go1;  // per-group continue decisions (written by one thread, read by all after a barrier)
    float bc[4];
    float wsum[4];
    float bsm[kC];
    float eneg[kC];
};

constexpr size_t kTileBytes = (size_t)kStages * 3 * kTile + kTile;  // Q,K,V per stage + P
constexpr size_t kTcSmemBytes = 232448;                            // the sm_100 per-block maximum

__device__ __forceinline__ void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory"); }

__device__ __forceinline__ void report(int *err, int *abort_flag, int code) {
    *(volatile int *)abort_flag = 1;
    if (err) atomicExch(err, (int)(kErrMagic | (uint32_t)code));
}

// bf16x8 in a uint4 scaled by s, rounded back to bf16 (nearest even)
__device__ __forceinline__ uint4 scale_bf16x8(uint4 u, float s) {
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float lo = __uint_as_float(w[i] << 16) * s;
        float hi = __uint_as_float(w[i] & 0xFFFF0000u) * s;
        __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
        w[i] = *reinterpret_cast<uint32_t *>(&h2);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h2);
}

// Scale row r of a 128 x 128 swizzled bf16 tile in place.
__device__ __forceinline__ void scale_row_inplace(uint8_t *tile, int r, float s) {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        uint32_t off = (uint32_t)(c >> 3) * kHalf + (uint32_t)r * 128u + (uint32_t)(((c & 7) ^ (r & 7)) * 16);
        uint4 *p = reinterpret_cast<uint4 *>(tile + off);
        *p = scale_bf16x8(*p, s);
    }
}

template <int MODE>
__global__ void __launch_bounds__(kTcThreads, 1)
gret_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const float *__restrict__ logits, float inv_tau,
               bf16_t *__restrict__ o, const float *__restrict__ S_in, float *__restrict__ S_out,
               float *__restrict__ G_out, int N, int H, int seg_len, int P, int *err) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base_u32 = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (base_u32 & 1023u)) & 1023u;
    uint8_t *tiles = smem_raw + pad;
    TcSmem &sm = *reinterpret_cast<TcSmem *>(tiles + kTileBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (pad + kTileBytes + sizeof(TcSmem) > kTcSmemBytes) {  // cannot happen with a 16-B aligned window
        if (tid == 0 && err) atomicExch(err, (int)(kErrMagic | 9u));
        return;
    }
    const int p = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int t_begin = p * seg_len;
    const int t_end = min(N, t_begin + seg_len);
    const int nchunks = (t_end - t_begin + kC - 1) / kC;
    const size_t bhp = ((size_t)b * H + h) * P + p;
    uint8_t *Pbuf = tiles + (size_t)kStages * 3 * kTile;
    auto stage_q = [&](int s) { return tiles + (size_t)s * 3 * kTile; };
    auto stage_k = [&](int s) { return tiles + (size_t)s * 3 * kTile + kTile; };
    auto stage_v = [&](int s) { return tiles + (size_t)s * 3 * kTile + 2 * kTile; };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
            mbar_init(&sm.pq_ready[s], 1);
        }
        mbar_init(&sm.as_full, 1);
        mbar_init(&sm.as_free, 1);
        mbar_init(&sm.o_full, 1);
        mbar_init(&sm.o_free, 1);
        mbar_init(&sm.u_full, 1);
        mbar_init(&sm.u_free, 1);
        mbar_init(&sm.s_ready, 1);
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    volatile int *abort_flag = &sm.abort_flag;

    // chunk order: OUTPUT forwards, SEG_STATE backwards (running suffix decay)
    auto chunk_start = [&](int i) {
        int c = (MODE == MODE_OUTPUT) ? i : (nchunks - 1 - i);
        return t_begin + c * kC;
    };

    if (warp == 8) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            if (MODE == MODE_OUTPUT) tma_prefetch_desc(&tm_q);
            const uint32_t bytes = (MODE == MODE_OUTPUT) ? 3 * kTile : 2 * kTile;
            for (int i = 0; i < nchunks; ++i) {
                const int s = i % kStages;
                if (i >= kStages && !mbar_wait(&sm.empty[s], ((i / kStages) + 1) & 1, abort_flag)) {
                    report(err, &sm.abort_flag, 1);
                    break;
                }
                const int n0 = chunk_start(i);
                mbar_arrive_expect_tx(&sm.full[s], bytes);
                for (int half = 0; half < 2; ++half) {
                    if (MODE == MODE_OUTPUT) tma_load_4d(stage_q(s) + half * kHalf, &tm_q, &sm.full[s], half * 64, h, n0, b);
                    tma_load_4d(stage_k(s) + half * kHalf, &tm_k, &sm.full[s], half * 64, h, n0, b);
                    tma_load_4d(stage_v(s) + half * kHalf, &tm_v, &sm.full[s], half * 64, h, n0, b);
                }
            }
            // leave no copy in flight: wait for the last loads of each stage
            for (int i = max(0, nchunks - kStages); i < nchunks; ++i)
                mbar_wait(&sm.full[i % kStages], (i / kStages) & 1, abort_flag, 200000000ull);
        }
    } else if (warp == 9) {
        // --------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_qk = idesc_bf16_f32(kC, kC, false, false);   // A=Q (K-major), B=K (K-major)
            const uint32_t id_vp = idesc_bf16_f32(kD, kC, true, false);    // A=V^T (MN-major), B=P (K-major)
            const uint32_t id_sq = idesc_bf16_f32(kD, kC, false, false);   // A=S^T (TMEM), B=Q' (K-major)
            const uint32_t id_vk = idesc_bf16_f32(kD, kD, true, true);     // A=V^T (MN-major), B=K' (MN-major)
            bool ok = true;
            for (int i = 0; i < nchunks && ok; ++i) {
                const int s = i % kStages;
                const uint32_t q_a = smem_u32(stage_q(s)), k_a = smem_u32(stage_k(s)), v_a = smem_u32(stage_v(s));
                ok = mbar_wait(&sm.full[s], (i / kStages) & 1, abort_flag);
                if (!ok) break;
                if (MODE == MODE_OUTPUT) {
                    if (i > 0 && !(ok = mbar_wait(&sm.as_free, (i - 1) & 1, abort_flag))) break;
                    tc_fence_after();
                    for (int kk = 0; kk < 8; ++kk) {  // MMA1: A = Q K^T
                        const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                        mma_ss(tmem + kColA, smem_desc_sw128(q_a + off, 16, 1024), smem_desc_sw128(k_a + off, 16, 1024),
                               id_qk, kk > 0);
                    }
                    mma_commit(&sm.as_full);
                }
                if (!(ok = mbar_wait(&sm.pq_ready[s], (i / kStages) & 1, abort_flag))) break;
                tc_fence_after();
                if (MODE == MODE_OUTPUT) {
                    if (i > 0 && !(ok = mbar_wait(&sm.o_free, (i - 1) & 1, abort_flag))) break;
                    tc_fence_after();
                    const uint32_t p_a = smem_u32(Pbuf);
                    for (int kk = 0; kk < 8; ++kk) {  // MMA2: O^T = V^T P^T
                        mma_ss(tmem + kColO, smem_desc_sw128(v_a + kk * 2048, kHalf, 1024),
                               smem_desc_sw128(p_a + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024), id_vp, kk > 0);
                    }
                    if (!(ok = mbar_wait(&sm.s_ready, i & 1, abort_flag))) break;
                    tc_fence_after();
                    for (int kk = 0; kk < 8; ++kk) {  // MMA3: O^T += S^T Q'^T
                        const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                        mma_ts(tmem + kColO, tmem + kColS + kk * 8, smem_desc_sw128(q_a + off, 16, 1024), id_sq, 1);
                    }
                    mma_commit(&sm.o_full);
                    if (i > 0 && !(ok = mbar_wait(&sm.u_free, (i - 1) & 1, abort_flag))) break;
                    tc_fence_after();
                }
                for (int kk = 0; kk < 8; ++kk) {  // MMA4: U^T (+)= V^T K'
                    const uint32_t acc = (MODE == MODE_OUTPUT) ? (kk > 0) : (i > 0 || kk > 0);
                    mma_ss(tmem + kColU, smem_desc_sw128(v_a + kk * 2048, kHalf, 1024),
                           smem_desc_sw128(k_a + kk * 2048, kHalf, 1024), id_vk, acc);
                }
                if (MODE == MODE_OUTPUT) mma_commit(&sm.u_full);
                mma_commit(&sm.empty[s]);
            }
            if (!ok) report(err, &sm.abort_flag, 2);
            if (MODE == MODE_SEG_STATE) mma_commit(&sm.u_full);
            // drain: nothing of ours may still run when TMEM is released
            mma_commit(&sm.drain);
            mbar_wait(&sm.drain, 0, abort_flag, 200000000ull);
        }
    } else if (warp >= 4) {
        // ------------------------------------ decay, P and in-place scaling
        const int j = tid - 128;  // token row of the chunk, TMEM lane j
        const int w4 = warp - 4;
        const uint32_t lane_base = (uint32_t)(w4 * 32) << 16;
        float suffix = 0.f;  // SEG_STATE: log decay of the chunks already processed (after this one)
        for (int i = 0; i < nchunks; ++i) {
            const int s = i % kStages;
            const int n0 = chunk_start(i);
            const int len = min(kC, N - n0);
            // chunk-local inclusive cumsum of log gates
            float lg = (j < len) ? log_gate(logits[((size_t)b * N + n0 + j) * H + h], inv_tau) : 0.f;
            float x = lg;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                float y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            if (lane == 31) sm.wsum[w4] = x;
            named_bar(1, 128);
            float pre = 0.f;
            for (int w = 0; w < w4; ++w) pre += sm.wsum[w];
            const float bj = x + pre;
            const float bC = sm.wsum[0] + sm.wsum[1] + sm.wsum[2] + sm.wsum[3];
            sm.bsm[j] = bj;
            const bool factor = (bC > -80.f);  // e^{-b_k} stays finite: use e^{b_j} e^{-b_k}
            sm.eneg[j] = factor ? __expf(-bj) : 0.f;
            named_bar(1, 128);  // bsm / eneg complete; wsum may be reused next chunk

            bool ok = true;
            if (MODE == MODE_OUTPUT) {
                if (j == 0) {
                    ok = mbar_wait(&sm.as_full, i & 1, abort_flag);
                    if (ok && i > 0) ok = mbar_wait(&sm.o_full, (i - 1) & 1, abort_flag);  // MMA2(i-1) done with P
                    if (!ok) report(err, &sm.abort_flag, 3);
                    sm.go1 = ok && !*abort_flag;
                }
                named_bar(1, 128);
                if (!sm.go1) break;
                tc_fence_after();
                const float ebj = __expf(bj);
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t r[32];
                    tmem_ld32(tmem + kColA + lane_base + cb * 32, r);
                    tmem_wait_ld();
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int k0 = cb * 32 + 2 * e;
                        float v0 = 0.f, v1 = 0.f;
                        if (k0 <= j) v0 = __uint_as_float(r[2 * e]) * (factor ? ebj * sm.eneg[k0] : __expf(bj - sm.bsm[k0]));
                        if (k0 + 1 <= j)
                            v1 = __uint_as_float(r[2 * e + 1]) * (factor ? ebj * sm.eneg[k0 + 1] : __expf(bj - sm.bsm[k0 + 1]));
                        pk[e] = pack_bf16x2(v0, v1);
                    }
                    // keys cb*32 .. cb*32+31 -> 4 chunks of 16 B in row j of P
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int key = cb * 32 + q4 * 8;
                        const uint32_t off = (uint32_t)(key >> 6) * kHalf + (uint32_t)j * 128u +
                                             (uint32_t)((((key & 63) >> 3) ^ (j & 7)) * 16);
                        *reinterpret_cast<uint4 *>(Pbuf + off) =
                            make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
                    }
                }
                tc_fence_before();
                scale_row_inplace(stage_q(s), j, ebj);          // Q'_j = e^{b_j} q_j
                scale_row_inplace(stage_k(s), j, __expf(bC - bj));  // K'_j = e^{b_C - b_j} k_j
            } else {
                if (j == 0) {
                    ok = mbar_wait(&sm.full[s], (i / kStages) & 1, abort_flag);
                    if (!ok) report(err, &sm.abort_flag, 3);
                    sm.go1 = ok && !*abort_flag;
                }
                named_bar(1, 128);
                if (!sm.go1) break;
                // weight of token j: decay from j to the segment end
                scale_row_inplace(stage_k(s), j, __expf(suffix + (bC - bj)));
                suffix += bC;
            }
            fence_proxy_async_smem();
            if (MODE == MODE_OUTPUT && j == 0) sm.bc[i & 3] = bC;
            named_bar(1, 128);
            if (j == 0) {
                if (MODE == MODE_OUTPUT) mbar_arrive(&sm.as_free);
                mbar_arrive(&sm.pq_ready[s]);
            }
        }
        if (MODE == MODE_SEG_STATE && j == 0 && G_out) G_out[bhp] = suffix;
    } else {
        // ------------------------------------------- state warps + output
        const int c = tid;  // d_v column = TMEM lane
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        if (MODE == MODE_OUTPUT) {
            float S[kD];  // S^T row c: S[i] = S[i][c]
#pragma unroll
            for (int i = 0; i < kD; ++i) S[i] = S_in ? S_in[bhp * kD * kD + (size_t)i * kD + c] : 0.f;
            auto put_state = [&]() {  // bf16 S^T into TMEM columns kColS.. (A operand of MMA3)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(S[32 * q + 2 * e], S[32 * q + 2 * e + 1]);
                    tmem_st16(tmem + kColS + lane_base + 16 * q, pk);
                }
                tmem_wait_st();
                tc_fence_before();
            };
            put_state();
            named_bar(2, 128);
            if (c == 0) mbar_arrive(&sm.s_ready);
            for (int i = 0; i < nchunks; ++i) {
                const int n0 = chunk_start(i);
                const int len = min(kC, N - n0);
                bool ok = true;
                if (c == 0) {
                    ok = mbar_wait(&sm.u_full, i & 1, abort_flag);
                    if (!ok) report(err, &sm.abort_flag, 4);
                    sm.go0 = ok && !*abort_flag;
                }
                named_bar(2, 128);
                if (!sm.go0) break;
                tc_fence_after();
                const float ebC = __expf(sm.bc[i & 3]);
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t r[32];
                    tmem_ld32(tmem + kColU + lane_base + cb * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) S[cb * 32 + e] = fmaf(ebC, S[cb * 32 + e], __uint_as_float(r[e]));
                }
                tc_fence_before();
                named_bar(2, 128);
                if (c == 0) mbar_arrive(&sm.u_free);
                if (i + 1 < nchunks) {
                    put_state();
                    named_bar(2, 128);
                    if (c == 0) mbar_arrive(&sm.s_ready);
                }
                // output rows of this chunk: o[n0 + j][c] = O^T[c][j]
                tc_fence_after();
                bf16_t *ocol = o + (((size_t)b * N + n0) * H + h) * kD + c;
                const size_t rstride = (size_t)H * kD;
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t r[32];
                    tmem_ld32(tmem + kColO + lane_base + cb * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int jq = cb * 32 + e;
                        if (jq < len) ocol[(size_t)jq * rstride] = from_f32<bf16_t>(__uint_as_float(r[e]));
                    }
                }
                tc_fence_before();
                named_bar(2, 128);
                if (c == 0) mbar_arrive(&sm.o_free);
            }
            named_bar(2, 128);
            if (c == 0) sm.go0 = !*abort_flag;
            named_bar(2, 128);
            if (S_out && sm.go0) {
#pragma unroll
                for (int i = 0; i < kD; ++i) S_out[bhp * kD * kD + (size_t)i * kD + c] = S[i];
            }
        } else {
            bool ok = true;
            if (c == 0) {
                ok = mbar_wait(&sm.u_full, 0, abort_flag, 4000000000ull);
                if (!ok) report(err, &sm.abort_flag, 5);
                sm.go0 = ok && !*abort_flag;
            }
            named_bar(2, 128);
            if (sm.go0) {
                tc_fence_after();
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t r[32];
                    tmem_ld32(tmem + kColU + lane_base + cb * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        S_out[bhp * kD * kD + (size_t)(cb * 32 + e) * kD + c] = __uint_as_float(r[e]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace yoco

// ------------------------------------------------------------------ host side
namespace yoco_host {
using namespace yoco;

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// [B, N, H, 128] bf16 as a 4-D map {d, h, n, b}; box {64, 1, 128, 1}, 128-B swizzle
static bool make_map(CUtensorMap *m, const void *ptr, int B, int N, int H) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2, (cuuint64_t)N * H * kD * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)kC, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool gret_tc_eligible(int B, int N, int H, int dk, int dv, yoco_dtype dt) {
    return dt == YOCO_BF16 && dk == kD && dv == kD && N >= 1 && B >= 1 && H >= 1 && B <= 65535 && H <= 65535;
}

static int tc_segments(int B, int N, int H) {
    const int chunks = (N + kC - 1) / kC;
    int P = 152 / (B * H);
    if (P < 1) P = 1;
    if (P > chunks) P = chunks;
    return P;
}

static int tc_seg_len(int N, int P) {
    const int chunks = (N + kC - 1) / kC;
    return ((chunks + P - 1) / P) * kC;
}

size_t gret_tc_workspace(int B, int N, int H, int dk, int dv) {
    (void)dk; (void)dv;
    int P = tc_segments(B, N, H);
    size_t ws = 256;  // status word
    if (P > 1) ws += ((size_t)B * H * P * kD * kD + (size_t)B * H * P) * sizeof(float);
    return ws;
}

cudaError_t gret_prefill_tc(const GretArgs &a, void *ws, cudaStream_t st) {
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, a.q, a.B, a.N, a.H) || !make_map(&mk, a.k, a.B, a.N, a.H) || !make_map(&mv, a.v, a.B, a.N, a.H))
        return cudaErrorInvalidValue;
    int P = tc_segments(a.B, a.N, a.H);
    const int seg_len = tc_seg_len(a.N, P);
    P = (a.N + seg_len - 1) / seg_len;
    int *err = (int *)ws;
    float *E = (float *)((char *)ws + 256);
    float *G = E + (size_t)a.B * a.H * P * kD * kD;
    const float inv_tau = 1.0f / a.tau;
    cudaError_t e;
    e = cudaFuncSetAttribute(gret_tc_kernel<MODE_OUTPUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gret_tc_kernel<MODE_SEG_STATE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kTcSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(P, a.H, a.B);
    if (P == 1) {
        count_launches(1);
        gret_tc_kernel<MODE_OUTPUT><<<grid, kTcThreads, kTcSmemBytes, st>>>(
            mq, mk, mv, a.logits, inv_tau, (bf16_t *)a.o, a.state, a.state, nullptr, a.N, a.H, seg_len, 1, err);
        return cudaGetLastError();
    }
    count_launches(3);
    gret_tc_kernel<MODE_SEG_STATE><<<grid, kTcThreads, kTcSmemBytes, st>>>(
        mq, mk, mv, a.logits, inv_tau, nullptr, nullptr, E, G, a.N, a.H, seg_len, P, err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = gret_scan_launch(E, G, a.state, a.B * a.H, P, kD * kD, st)) != cudaSuccess) return e;
    gret_tc_kernel<MODE_OUTPUT><<<grid, kTcThreads, kTcSmemBytes, st>>>(
        mq, mk, mv, a.logits, inv_tau, (bf16_t *)a.o, E, nullptr, nullptr, a.N, a.H, seg_len, P, err);
    return cudaGetLastError();
}

}  // namespace yoco_host
