// gret_tc.cu -- chunkwise gated retention on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA), bf16 inputs, head size 128, 128-token chunks.
//
// Math (paper Section 3.1, Eq. 6 with consistent indices; Appendix F
// ChunkwiseRetention).  For a chunk with chunk-local cumulative log decay b_j
// (b_j = sum of log gamma over the chunk's tokens up to and including j) and the
// state S (d_k x d_v) before the chunk:
//     o_j  = sum_{k<=j} (q_j . k_k) e^{b_j - b_k} v_k  +  e^{b_j} q_j S
//     S'   = e^{b_C} S + sum_k e^{b_C - b_k} k_k^T v_k
// On the tensor cores, per chunk (lane = TMEM lane):
//     A    = Q K^T                               MMA1   lane = query j
//     P_jk = A_jk e^{-b_k} [k <= j]  (bf16, written over A in TMEM)
//     O    = P V + Q S                           MMA2 (P from TMEM), MMA3
//     o_j  = e^{b_j} O_j                         epilogue
//     U    = K'^T V,  K'_k = e^{b_C - b_k} k_k   MMA4   lane = d_k row i
//     S'   = e^{b_C} S + U   (fp32, registers of the state warps; bf16 copy in
//                             shared memory is MMA3's B operand)
// Factoring e^{b_j - b_k} = e^{b_j} e^{-b_k} needs e^{-b_k} finite; a chunk whose
// total log decay is below -60 instead multiplies P by e^{b_j - b_k} directly and
// scales Q's rows by e^{b_j} in place (and the epilogue multiplies by 1).
//
// Sequence parallelism: the sequence of every (b, h) is cut into P segments of
// whole chunks.  The segment-state kernel (gret_seg_kernel) walks a segment
// backwards and accumulates its zero-start end state
// E^T = sum_k e^{(decay after k to segment end)} v_k^T k_k directly in TMEM (every
// weight <= 1), plus the segment's total log decay.  An output CTA (gret_tc_kernel)
// then folds the earlier segments' end states into its initial state
// (S_start(p) = e^{G_{p-1}} S_start(p-1) + E_{p-1}) and runs the chunk recurrence
// above from it.  The last segment's end state is the call's final state, so the
// segment-state grid covers P-1 segments only.  With B*H >= #SMs, P = 1 and only the
// output kernel runs.
//
// Negligible weights are dropped (kDropLog): the backward walk of a segment stops at
// the first chunk whose newest token already carries a weight below e^-40 in the
// segment's end state (every older token's weight is smaller still), and the fold
// leaves out every earlier segment whose decay up to this segment's start is below
// e^-40.  What is left out is bounded by e^-40 ~ 4e-18 times the dropped terms'
// magnitudes.  With no decay (gamma = 1) nothing is dropped and the walk and the fold
// cover everything.  No CTA ever waits for another one: each output CTA folds the
// states it needs on its own, and the final state reaches `state` through a
// two-party hand-off (whichever of segment 0 and the last segment comes second
// writes it).
//
// Warp roles (320 threads): warps 0-3 keep the state (thread t = TMEM lane t =
// d_k row t), warps 4-7 compute the decay, P, the in-place scaling of K (and Q)
// and write the output rows (thread j = query row j), warp 8 issues TMA loads,
// warp 9 issues the MMAs: per chunk MMA1, then (factored chunks) MMA3 while P is
// being computed, then MMA4 so the state warps can start, then MMA2.
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
constexpr int kStages = 2;                  // OUTPUT: 2 x (Q, K, V)
constexpr int kTcThreads = 512;                 // 4 warpgroups: state, decay, TMA + MMA, epilogue
constexpr float kFactorMin = -60.f;         // chunk decay above which e^{-b_k} is used
constexpr float kDropLog = 40.f;            // state contributions weighted below e^-40 are left out

// Hand-off word per (b, h) for the final state (cleared by the segment-state grid):
constexpr int kHandInitRead = 1;            // segment 0 holds the caller's initial state
constexpr int kHandParked = 2;              // the last segment parked the final state in slot P

// TMEM columns: A / P, two O accumulators, U
constexpr uint32_t kColA = 0, kColO = 128, kColU = 384;


struct TcSmem {
    uint64_t full[kStages], empty[kStages], pq_ready[kStages], o_free[2], bc_ready[2], o_full[2];
    uint64_t full_v[kStages], o_staged[kStages], k_ready[kStages];
    uint64_t as_full, p_free, u_full, u_free, s_ready, drain;
    uint32_t tmem_base;
    int abort_flag;
    int go0, go1, go2;  // per-group continue decisions (written by one thread, read by all after a barrier)
    int hand_old;  // the final-state hand-off word as one thread saw it
    float wsum0[4], wsum1[4], wsum2[4];
    float gnw[kD], gnb[kD];  // GroupNorm affine of this head (output with Eq. 7 only)
    float bcr[4];  // chunk total log decay b_C, ring over chunks
    alignas(16) float ew[kC];  // e^{-b_k} (factored chunks) or b_k (direct chunks); read as float4

};

static_assert(offsetof(TcSmem, ew) % 16 == 0, "ew is read as float4");
constexpr size_t kTileBytes = (size_t)kStages * 3 * kTile + kTile;  // Q,K,V per stage + bf16 state
constexpr size_t kTcSmemBytes = 232448;                            // the sm_100 per-block maximum
static_assert(kTileBytes + sizeof(TcSmem) + 1024 <= kTcSmemBytes, "tiles + control block + alignment slack must fit");

// Named barrier of n threads.  bar.sync is the aligned form: all 32 lanes of a warp
// must execute it together, and nothing else makes a warp reconverge after one lane
// has waited alone (the `if (t == 0) { bounded wait }` pattern), so the warp is
// synchronised first.
__device__ __forceinline__ void named_bar(int id, int n) {
    __syncwarp();
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void report(int *err, int *abort_flag, int code) {
    *(volatile int *)abort_flag = 1;
    if (err) atomicExch(err, (int)(kErrMagic | (uint32_t)code));
}

// tanh on the special-function unit (the PTX approximate instruction, max relative
// error about 2^-11)
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// bf16x8 in a uint4 times the bf16 pair s2 (packed bf16x2 multiply, nearest even)
__device__ __forceinline__ uint4 scale_bf16x8(uint4 u, __nv_bfloat162 s2) {
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __hmul2(h[i], s2);
    return u;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h2);
}

// Byte offset of 16-B chunk c (0..15, 8 bf16 each) of row r in a 128 x 128
// swizzled bf16 tile ([64-column block][128 rows][128 B], chunks XOR row % 8).
__device__ __forceinline__ uint32_t tile_chunk(int r, int c) {
    return (uint32_t)(c >> 3) * kHalf + (uint32_t)r * 128u + (uint32_t)(((c & 7) ^ (r & 7)) * 16);
}

// Scale row r of a 128 x 128 swizzled bf16 tile in place.
__device__ __forceinline__ void scale_row_inplace(uint8_t *tile, int r, float s) {
    const __nv_bfloat162 s2 = __float2bfloat162_rn(s);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        uint4 *p = reinterpret_cast<uint4 *>(tile + tile_chunk(r, c));
        *p = scale_bf16x8(*p, s2);
    }
}

// Inclusive cumsum of one value per thread over a 128-thread group (4 warps).
__device__ __forceinline__ float group_scan(float x, float *wsum, int lane, int wq, int bar_id, float &total) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        float y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) wsum[wq] = x;
    named_bar(bar_id, 128);
    float pre = 0.f;
    for (int w = 0; w < wq; ++w) pre += wsum[w];
    total = wsum[0] + wsum[1] + wsum[2] + wsum[3];
    return x + pre;
}

// Initial state of segment p >= 1 of one (b, h): columns [OFF, OFF + 64) of row t
// (into S[OFF .. OFF + 63]):
//     S_start(p) = sum_{q<p} e^{dec(q)} E_q + e^{dec(-1)} S_init,  dec(q) = sum_{q<r<p} G_r,
// evaluated as the fold S <- e^{G_q} S + E_q in order of q, starting at the earliest
// segment q0 whose decay up to segment p is still >= e^-kDropLog (from S_init when
// even the caller's state is that close, else from zero).  E slots per (b, h):
// 0 .. P-2 the segments' end states, P-1 a copy of the caller's state.  The state
// warps fold columns 0-63 and the decay warps 64-127 of the same rows; every thread
// reads the same G values, so the loop bounds are uniform.
template <int OFF>
__device__ __forceinline__ void seg_initial_half(float (&S)[kD], const float *E, const float *G, size_t bh, int P,
                                                 int p, int t) {
    const float *g_bh = G + bh * P;
    float dec = 0.f;  // dec(q0)
    int q0 = p - 1;
    while (q0 > 0) {
        const float nd = dec + __ldcg(g_bh + q0);
        if (nd < -kDropLog) break;
        dec = nd;
        --q0;
    }
    const bool with_init = (q0 == 0) && (dec + __ldcg(g_bh) >= -kDropLog);
    const size_t slot0 = bh * (size_t)(P + 1);
#pragma unroll
    for (int c = 0; c < 64; ++c) S[OFF + c] = 0.f;
    if (!YOCO_DCHECK(slot0 + P < (size_t)(gridDim.x / P) * (P + 1), 0x40)) return;
    auto fold = [&](size_t slot, float gq) {  // S <- gq S + E_slot, 32 columns per round of loads
        const float4 *src = reinterpret_cast<const float4 *>(E + slot * kD * kD + (size_t)t * kD + OFF);
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
            float4 x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) x[u] = __ldcg(src + cb * 8 + u);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                float *s4 = &S[OFF + cb * 32 + 4 * u];
                s4[0] = fmaf(gq, s4[0], x[u].x);
                s4[1] = fmaf(gq, s4[1], x[u].y);
                s4[2] = fmaf(gq, s4[2], x[u].z);
                s4[3] = fmaf(gq, s4[3], x[u].w);
            }
        }
    };
    if (with_init) fold(slot0 + P - 1, 0.f);
    for (int q = q0; q < p; ++q) fold(slot0 + q, __expf(__ldcg(g_bh + q)));
}

template <int R>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(R)); }
template <int R>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(R)); }
// Registers per thread by warpgroup (launched with 128 each, 512 threads = the whole
// register file): state 216, decay 112, TMA + MMA 64, epilogue 120; 216 + 112 + 64 +
// 120 = 4 x 128, so the state warpgroup's increase is exactly what the others free
// (each does its decrease first thing).  With fewer for the TMA producer and the MMA
// issuer (48 or 56), values of their per-chunk loops lived in local memory, which
// misses L1 here (shared memory takes nearly all of it), and each reload cost an L2
// round trip on the pipeline's critical path; this split leaves no spill at all.
constexpr int kRegsState = 216, kRegsDecay = 112, kRegsIssue = 64, kRegsEpi = 120;
static_assert(kRegsState + kRegsDecay + kRegsIssue + kRegsEpi == 4 * 128, "the split must use the launch's registers");

// kGN: the epilogue applies the paper's Eq. 7 output (GroupNorm per head, then the
// swish gate) and writes z instead of the raw retention output o.
template <bool kGN>
__global__ void __launch_bounds__(kTcThreads, 1)
gret_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               const __grid_constant__ CUtensorMap tm_g,
               const float *__restrict__ logits, float inv_tau,
               float *__restrict__ state, float *__restrict__ E, float *__restrict__ G,
               int *__restrict__ hand, int N, int H, int seg_len, int P, int *err, uint64_t seg0_delay_ns,
               const bf16_t *__restrict__ gate, const float *__restrict__ gn_w, const float *__restrict__ gn_b,
               float gn_eps) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base_u32 = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (base_u32 & 1023u)) & 1023u;
    uint8_t *tiles = smem_raw + pad;
    TcSmem &sm = *reinterpret_cast<TcSmem *>(tiles + kTileBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int NS = kStages;
    if (pad + kTileBytes + sizeof(TcSmem) > kTcSmemBytes) {  // cannot happen with a 16-B aligned window
        if (tid == 0 && err) atomicExch(err, (int)(kErrMagic | 9u));
        return;
    }
    // segment-major linear grid: the segment-0 CTAs, which need nothing from the
    // segment-state grid, are dispatched first
    const int BH = (int)gridDim.x / P, r_bh = (int)blockIdx.x % BH;
    const int p = (int)blockIdx.x / BH, h = r_bh % H, b = r_bh / H;
    const int t_begin = p * seg_len;
    const int t_end = min(N, t_begin + seg_len);
    const int nchunks = (t_end - t_begin + kC - 1) / kC;
    const size_t bh = (size_t)b * H + h;  // E slots: bh * (P + 1) + q; G: bh * P + q
    // each stage holds Q, K, V of one chunk
    uint8_t *Sbuf = tiles + (size_t)6 * kTile;  // bf16 state, MMA3's B operand
    constexpr size_t kSS = 3 * (size_t)kTile;
    auto stage_q = [&](int s) { return tiles + (size_t)s * kSS; };
    auto stage_k = [&](int s) { return tiles + (size_t)s * kSS + kTile; };
    auto stage_v = [&](int s) { return stage_k(s) + kTile; };

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {  // ring barriers, one per stage
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
            mbar_init(&sm.pq_ready[s], 1);
        }
        for (int s = 0; s < 2; ++s) {  // double-buffered per-chunk barriers
            mbar_init(&sm.o_free[s], 1);
            mbar_init(&sm.bc_ready[s], 1);
            mbar_init(&sm.o_full[s], 1);
            mbar_init(&sm.full_v[s], 1);
            mbar_init(&sm.o_staged[s], 1);
            mbar_init(&sm.k_ready[s], 1);
        }
        mbar_init(&sm.as_full, 1);
        mbar_init(&sm.p_free, 1);
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
    // Programmatic dependent launch.  With P > 1 this grid is a dependent of the
    // segment-state grid, which waited for whatever ran before it before letting this
    // grid start: so the TMA producer reads q, k, v at once, and only E, G and the
    // state wait (state warps, segments p > 0).  This grid lets the next kernel (the
    // next call's segment-state grid) start its prologue on idle SMs right away; that
    // kernel waits too.
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    auto chunk_start = [&](int i) { return t_begin + i * kC; };
    auto chunk_log_gate = [&](int n0, int row) {
        return (n0 + row < N) ? log_gate(logits[((size_t)b * N + n0 + row) * H + h], inv_tau) : 0.f;
    };
    if (warp >= 8 && warp < 12) {
        regs_dec<kRegsIssue>();
        if (warp == 8) {
            // ------------------------------------------------------ TMA producer
            if (lane == 0) {
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_o);
                if (kGN) tma_prefetch_desc(&tm_g);
                // every q, k, v line is read once per pass and every o line written once:
                // all of them are marked first to leave L2 (measured: 0.235 -> 0.221 ms per
                // 32K x 24 x 128 layer; keeping the segment-state pass's k, v tiles for this
                // pass with evict-last was slower at every fraction of L2 tried)
                const uint64_t pol = l2_policy_evict_first();
                // Q and K complete `full`, V completes `full_v`.  The V slot doubles as the
                // staging buffer of the output rows of the chunk NS back: this thread stores
                // them (TMA) and waits for the store to read the slot before it loads the next
                // V there, so the state warps never wait on a store.
                auto store_out = [&](int c) {  // chunk c's staged output rows -> o
                    const int sc_ = c % NS;
                    if (!mbar_wait(&sm.o_staged[sc_], (c / NS) & 1, abort_flag)) {
                        report(err, &sm.abort_flag, 8);
                        return false;
                    }
                    const int nc = chunk_start(c);
                    tma_store_4d_hint(&tm_o, stage_v(sc_), 0, h, nc, b, pol);
                    tma_store_4d_hint(&tm_o, stage_v(sc_) + kHalf, 64, h, nc, b, pol);
                    bulk_commit_group();
                    return true;
                };
                for (int i = 0; i < nchunks; ++i) {
                    const int s = i % NS;
                    if (i >= NS && !mbar_wait(&sm.empty[s], ((i / NS) + 1) & 1, abort_flag)) {
                        report(err, &sm.abort_flag, 1);
                        break;
                    }
                    const int n0 = chunk_start(i);
                    mbar_arrive_expect_tx(&sm.full[s], 2 * kTile);
                    for (int half = 0; half < 2; ++half) {
                        tma_load_4d_hint(stage_k(s) + half * kHalf, &tm_k, &sm.full[s], half * 64, h, n0, b, pol);
                        tma_load_4d_hint(stage_q(s) + half * kHalf, &tm_q, &sm.full[s], half * 64, h, n0, b, pol);
                        // Eq. 7: the chunk's gate rows into L2, where the epilogue's own row
                        // loads find them about two chunks from now
                        if (kGN) tma_prefetch_l2_4d(&tm_g, half * 64, h, n0, b);
                    }
                    if (i >= NS) {
                        if (!store_out(i - NS)) break;
                        bulk_wait_read_all();  // the slot has been read: V(i) may land in it
                    }
                    mbar_arrive_expect_tx(&sm.full_v[s], kTile);
                    for (int half = 0; half < 2; ++half)
                        tma_load_4d_hint(stage_v(s) + half * kHalf, &tm_v, &sm.full_v[s], half * 64, h, n0, b, pol);
                }
                // leave no copy in flight: wait for the last loads of each stage
                for (int i = max(0, nchunks - NS); i < nchunks; ++i) {
                    mbar_wait(&sm.full[i % NS], (i / NS) & 1, abort_flag, 200000000ull);
                    mbar_wait(&sm.full_v[i % NS], (i / NS) & 1, abort_flag, 200000000ull);
                }
                // the output rows of the last NS chunks, then every store complete before exit
                for (int c = max(0, nchunks - NS); c < nchunks && !*abort_flag; ++c)
                    if (!store_out(c)) break;
                bulk_wait_all();
            }
        } else if (warp == 9) {
            // --------------------------------------------------------- MMA issuer
            if (lane == 0) {
                const uint32_t id_qk = idesc_bf16_f32(kC, kC, false, false);  // A=Q (K-major),    B=K (K-major)
                const uint32_t id_pv = idesc_bf16_f32(kC, kD, false, true);   // A=P (TMEM),       B=V (N-major)
                const uint32_t id_qs = idesc_bf16_f32(kC, kD, false, true);   // A=Q (K-major),    B=S (N-major)
                const uint32_t id_kv = idesc_bf16_f32(kD, kD, true, true);    // A=K'^T (M-major), B=V (N-major)
                bool ok = true;
                for (int i = 0; i < nchunks && ok; ++i) {
                    const int s = i % NS, ob = i & 1;
                    const uint32_t q_a = smem_u32(stage_q(s)), k_a = smem_u32(stage_k(s)), v_a = smem_u32(stage_v(s));
                    if (!(ok = mbar_wait(&sm.full[s], (i / NS) & 1, abort_flag))) break;
                    // P of the previous chunk (TMEM columns of A) must have been consumed
                    if (i > 0 && !(ok = mbar_wait(&sm.p_free, (i - 1) & 1, abort_flag))) break;
                    tc_fence_after();
                    for (int kk = 0; kk < 8; ++kk) {  // MMA1: A = Q K^T
                        const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                        mma_ss(tmem + kColA, smem_desc_sw128(q_a + off, 16, 1024), smem_desc_sw128(k_a + off, 16, 1024),
                               id_qk, kk > 0);
                    }
                    mma_commit(&sm.as_full);
                    // the decay warps publish the chunk's total decay first: it decides the order
                    if (!(ok = mbar_wait(&sm.bc_ready[i & 1], (i / 2) & 1, abort_flag))) break;
                    const bool factor = sm.bcr[i & 3] > kFactorMin;
                    if (i >= 2 && !(ok = mbar_wait(&sm.o_free[ob], ((i / 2) - 1) & 1, abort_flag))) break;
                    const uint32_t o_t = tmem + kColO + 128 * ob;
                    const uint32_t s_a = smem_u32(Sbuf);
                    auto mma3 = [&]() {  // O = Q S  (Q' = diag(e^b) Q in direct chunks)
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                            mma_ss(o_t, smem_desc_sw128(q_a + off, 16, 1024),
                                   smem_desc_sw128(s_a + kk * 2048, kHalf, 1024), id_qs, kk > 0);
                        }
                    };
                    if (!factor) {  // Q is rescaled in place together with P
                        if (!(ok = mbar_wait(&sm.pq_ready[s], (i / NS) & 1, abort_flag))) break;
                    }
                    // the cross term needs nothing else from the decay warps: it fills the P bubble
                    if (!(ok = mbar_wait(&sm.s_ready, i & 1, abort_flag))) break;
                    tc_fence_after();
                    mma3();
                    if (!(ok = mbar_wait(&sm.k_ready[s], (i / NS) & 1, abort_flag))) break;
                    if (!(ok = mbar_wait(&sm.full_v[s], (i / NS) & 1, abort_flag))) break;
                    if (i > 0 && !(ok = mbar_wait(&sm.u_free, (i - 1) & 1, abort_flag))) break;
                    tc_fence_after();
                    for (int kk = 0; kk < 8; ++kk)  // MMA4: U = K'^T V
                        mma_ss(tmem + kColU, smem_desc_sw128(k_a + kk * 2048, kHalf, 1024),
                               smem_desc_sw128(v_a + kk * 2048, kHalf, 1024), id_kv, kk > 0);
                    mma_commit(&sm.u_full);
                    if (factor) {
                        if (!(ok = mbar_wait(&sm.pq_ready[s], (i / NS) & 1, abort_flag))) break;
                        tc_fence_after();
                    }
                    for (int kk = 0; kk < 8; ++kk)  // MMA2: O += P V
                        mma_ts(o_t, tmem + kColA + kk * 8, smem_desc_sw128(v_a + kk * 2048, kHalf, 1024), id_pv, 1);
                    mma_commit(&sm.o_full[ob]);
                    mma_commit(&sm.p_free);
                    mma_commit(&sm.empty[s]);
                }
                if (!ok) report(err, &sm.abort_flag, 2);
                // drain: nothing of ours may still run when TMEM is released
                mma_commit(&sm.drain);
                mbar_wait(&sm.drain, 0, abort_flag, 200000000ull);
            }
        }
    } else if (warp >= 12) {
        regs_dec<kRegsEpi>();
        // ----------------------------------------------------- epilogue warps
        // Output rows o_j = e^{b_j} O_j (or O_j in direct chunks), staged as bf16 in
        // the chunk's V slot (free once MMA2 is done); the TMA producer thread stores
        // them.  With kGN, Eq. 7's output instead: z_j = swish(g_j) (.)
        // (w (.) (o_j - mean_j) / sqrt(var_j + eps) + b), the moments over the head's
        // 128 channels of the fp32 row; the gate row is requested before the wait for
        // O, so it lands meanwhile.  Thread j = TMEM lane j = query row j.
        const int j = tid - 384;
        const int wq = warp - 12;
        const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
        if (kGN) {  // this head's affine, identity when absent
            sm.gnw[j] = gn_w ? gn_w[(size_t)h * kD + j] : 1.f;
            sm.gnb[j] = gn_b ? gn_b[(size_t)h * kD + j] : 0.f;
            named_bar(3, 128);
        }
        float lg_next = (nchunks > 0) ? chunk_log_gate(chunk_start(0), j) : 0.f;
        for (int i = 0; i < nchunks; ++i) {
            const int s = i % NS;
            float bC;
            const float bj = group_scan(lg_next, sm.wsum2, lane, wq, 3, bC);
            if (i + 1 < nchunks) lg_next = chunk_log_gate(chunk_start(i + 1), j);
            const float sc = (bC > kFactorMin) ? __expf(bj) : 1.f;  // output row scale
            // kGN: swish(g) = g sigmoid(g) of this row's gate, as bf16 pairs, worked out
            // before O is ready (sigmoid(x) = (1 + tanh(x / 2)) / 2)
            uint32_t sw[kGN ? kD / 2 : 1];
            if (kGN) {
                const int n = chunk_start(i) + j;
                const uint4 *src = reinterpret_cast<const uint4 *>(gate + (((size_t)b * N + n) * H + h) * kD);
#pragma unroll
                for (int c = 0; c < kD / 8; ++c) {
                    const uint4 u = (n < N) ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
                    sw[4 * c] = u.x; sw[4 * c + 1] = u.y; sw[4 * c + 2] = u.z; sw[4 * c + 3] = u.w;
                }
#pragma unroll
                for (int c2 = 0; c2 < kD / 2; ++c2) {
                    const float h0 = 0.5f * __uint_as_float(sw[c2] << 16);
                    const float h1 = 0.5f * __uint_as_float(sw[c2] & 0xFFFF0000u);
                    sw[c2] = pack_bf16x2(fmaf(h0, tanh_approx(h0), h0), fmaf(h1, tanh_approx(h1), h1));
                }
            }
            if (j == 0) {
                const bool ok = mbar_wait(&sm.o_full[i & 1], (i / 2) & 1, abort_flag);
                if (!ok) report(err, &sm.abort_flag, 6);
                sm.go2 = ok && !*abort_flag;
            }
            named_bar(3, 128);
            if (!sm.go2) break;
            tc_fence_after();
            uint8_t *stage_o = stage_v(s);
            const uint32_t o_t = tmem + kColO + 128 * (i & 1) + lane_base;
            if (!kGN) {
                const uint64_t sc2 = f2_pack(sc, sc);
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t r[32];
                    tmem_ld32(o_t + cb * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {  // two columns per packed multiply
                            float y0, y1;
                            f2_unpack(f2_mul(f2_pack(__uint_as_float(r[8 * q4 + 2 * e]),
                                                     __uint_as_float(r[8 * q4 + 2 * e + 1])), sc2), y0, y1);
                            w[e] = pack_bf16x2(y0, y1);
                        }
                        *reinterpret_cast<uint4 *>(stage_o + tile_chunk(j, cb * 4 + q4)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            } else {
                // moments of the fp32 row x = sc O about its first element (one pass
                // over O in tensor memory, packed pairs), then the output pass:
                //   z = swish(g) (w ((x - mean) / sqrt(var + eps)) + b)
                //     = swish(g) (w (O a + c) + b),  a = sc / sqrt(var + eps), c = -mean / sqrt(var + eps)
                float o0;
                {
                    uint32_t r0[1];
                    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n" : "=r"(r0[0]) : "r"(o_t));
                    tmem_wait_ld();
                    o0 = __uint_as_float(r0[0]);
                }
                const uint64_t shift2 = f2_pack(-o0, -o0), one2 = f2_pack(1.f, 1.f);
                uint64_t sum2 = 0, sq2 = 0;  // (0.f, 0.f)
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t r[32];
                    tmem_ld32(o_t + cb * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const uint64_t dv = f2_add(f2_pack(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), shift2);
                        sum2 = f2_fma(dv, one2, sum2);
                        sq2 = f2_fma(dv, dv, sq2);
                    }
                }
                float s0, s1, q0, q1;
                f2_unpack(sum2, s0, s1);
                f2_unpack(sq2, q0, q1);
                const float md = (s0 + s1) * (1.f / kD);                    // mean of O - o0
                const float var = sc * sc * fmaxf((q0 + q1) * (1.f / kD) - md * md, 0.f);
                const float rstd = rsqrtf(var + gn_eps);
                const float a = sc * rstd, c = -(sc * (o0 + md)) * rstd;
                const uint64_t a2 = f2_pack(a, a), c2 = f2_pack(c, c);
                const bool affine = (gn_w != nullptr) || (gn_b != nullptr);
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t r[32];
                    tmem_ld32(o_t + cb * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int col = cb * 32 + 8 * q4 + 2 * e;
                            uint64_t y = f2_fma(f2_pack(__uint_as_float(r[8 * q4 + 2 * e]),
                                                        __uint_as_float(r[8 * q4 + 2 * e + 1])), a2, c2);
                            if (affine)
                                y = f2_fma(y, f2_pack(sm.gnw[col], sm.gnw[col + 1]), f2_pack(sm.gnb[col], sm.gnb[col + 1]));
                            const uint32_t s2 = sw[col / 2];
                            float z0, z1;
                            f2_unpack(f2_mul(y, f2_pack(__uint_as_float(s2 << 16), __uint_as_float(s2 & 0xFFFF0000u))),
                                      z0, z1);
                            w[e] = pack_bf16x2(z0, z1);
                        }
                        *reinterpret_cast<uint4 *>(stage_o + tile_chunk(j, cb * 4 + q4)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            named_bar(3, 128);
            if (j == 0) {
                mbar_arrive(&sm.o_free[i & 1]);
                mbar_arrive(&sm.o_staged[s]);  // the TMA producer stores the rows
            }
        }
    } else if (warp >= 4) {
        regs_dec<kRegsDecay>();
        // ------------------------------ decay, P, in-place scaling of K (and Q)
        const int j = tid - 128;  // token row of the chunk = TMEM lane
        const int wq = warp - 4;
        const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
        if (p > 0) {  // columns 64-127 of row j of this segment's initial state, for the state warps
            float Sh[kD];
            asm volatile("griddepcontrol.wait;\n" ::: "memory");
            seg_initial_half<64>(Sh, E, G, bh, P, p, j);
            float4 *hi = reinterpret_cast<float4 *>(Sbuf + (size_t)j * 256);
#pragma unroll
            for (int c4 = 0; c4 < 16; ++c4)
                hi[c4] = make_float4(Sh[64 + 4 * c4], Sh[64 + 4 * c4 + 1], Sh[64 + 4 * c4 + 2], Sh[64 + 4 * c4 + 3]);
            named_bar(4, 256);
        }
        float lg_next = (nchunks > 0) ? chunk_log_gate(chunk_start(0), j) : 0.f;
        bool alive = true;
        for (int i = 0; i < nchunks && alive; ++i) {
            const int s = i % NS;
            float bC;
            const float bj = group_scan(lg_next, sm.wsum1, lane, wq, 1, bC);
            if (i + 1 < nchunks) lg_next = chunk_log_gate(chunk_start(i + 1), j);  // in flight during this chunk
            const bool factor = (bC > kFactorMin);
            sm.ew[j] = factor ? __expf(-bj) : bj;
            if (j == 0) {
                sm.bcr[i & 3] = bC;
                mbar_arrive(&sm.bc_ready[i & 1]);
            }
            named_bar(1, 128);  // ew complete; wsum1 free for the next chunk
            bool ok = true;
            if (j == 0) {
                ok = mbar_wait(&sm.as_full, i & 1, abort_flag);
                if (!ok) report(err, &sm.abort_flag, 3);
                sm.go1 = ok && !*abort_flag;
            }
            named_bar(1, 128);
            if (!sm.go1) {
                alive = false;
                break;
            }
            // K'_j = e^{b_C - b_j} k_j in place first: MMA4 and the state chain wait on it
            scale_row_inplace(stage_k(s), j, __expf(bC - bj));
            fence_proxy_async_smem();
            named_bar(1, 128);
            if (j == 0) mbar_arrive(&sm.k_ready[s]);
            tc_fence_after();
            // P row j over A row j, written in place as packed bf16 (keys 2c, 2c+1 in column c).
            // The 32 rows of warp wq end in key block wq: blocks before it need no mask,
            // blocks after it are zero and are not loaded.
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t pk[16];
                if (cb > wq) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) pk[e] = 0u;
                } else {
                    uint32_t r[32];
                    tmem_ld32(tmem + kColA + lane_base + cb * 32, r);
                    tmem_wait_ld();
                    if (factor && cb < wq) {
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const float4 w = *reinterpret_cast<const float4 *>(&sm.ew[cb * 32 + 4 * e4]);
                            float v0, v1, v2, v3;
                            f2_unpack(f2_mul(f2_pack(__uint_as_float(r[4 * e4]), __uint_as_float(r[4 * e4 + 1])),
                                             f2_pack(w.x, w.y)), v0, v1);
                            f2_unpack(f2_mul(f2_pack(__uint_as_float(r[4 * e4 + 2]), __uint_as_float(r[4 * e4 + 3])),
                                             f2_pack(w.z, w.w)), v2, v3);
                            pk[2 * e4] = pack_bf16x2(v0, v1);
                            pk[2 * e4 + 1] = pack_bf16x2(v2, v3);
                        }
                    } else if (factor) {
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const int k0 = cb * 32 + 4 * e4;
                            const float4 w = *reinterpret_cast<const float4 *>(&sm.ew[k0]);
                            const float v0 = (k0 <= j) ? __uint_as_float(r[4 * e4]) * w.x : 0.f;
                            const float v1 = (k0 + 1 <= j) ? __uint_as_float(r[4 * e4 + 1]) * w.y : 0.f;
                            const float v2 = (k0 + 2 <= j) ? __uint_as_float(r[4 * e4 + 2]) * w.z : 0.f;
                            const float v3 = (k0 + 3 <= j) ? __uint_as_float(r[4 * e4 + 3]) * w.w : 0.f;
                            pk[2 * e4] = pack_bf16x2(v0, v1);
                            pk[2 * e4 + 1] = pack_bf16x2(v2, v3);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int k0 = cb * 32 + 2 * e;
                            const float v0 = (k0 <= j) ? __uint_as_float(r[2 * e]) * __expf(bj - sm.ew[k0]) : 0.f;
                            const float v1 = (k0 + 1 <= j) ? __uint_as_float(r[2 * e + 1]) * __expf(bj - sm.ew[k0 + 1]) : 0.f;
                            pk[e] = pack_bf16x2(v0, v1);
                        }
                    }
                }
                tmem_st16(tmem + kColA + lane_base + cb * 16, pk);  // columns already read
            }
            tmem_wait_st();
            tc_fence_before();
            if (!factor) scale_row_inplace(stage_q(s), j, __expf(bj));  // Q'_j = e^{b_j} q_j
            fence_proxy_async_smem();
            named_bar(1, 128);
            if (j == 0) mbar_arrive(&sm.pq_ready[s]);
        }
    } else {
        regs_inc<kRegsState>();
        // ------------------------------------------------------- state warps
        const int t = tid;  // TMEM lane: d_k row t of S and U
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        float S[kD];  // row t of the state, fp32
        // Segment 0 starts from the caller's state and reads it directly, so it runs
        // alongside the segment-state grid; later segments wait for that grid and fold
        // the end states they need into their own initial state (row t each)
        if (p == 0) {
            if (seg0_delay_ns) {  // test hook: take the caller's state late (bounded by the host)
                uint64_t t0, tn;
                asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
                do {
                    __nanosleep(1000);
                    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(tn));
                } while (tn - t0 < seg0_delay_ns);
            }
            const float4 *src = reinterpret_cast<const float4 *>(state + bh * kD * kD + (size_t)t * kD);
#pragma unroll
            for (int c4 = 0; c4 < kD / 4; ++c4) {
                const float4 x = __ldcg(src + c4);
                S[4 * c4] = x.x; S[4 * c4 + 1] = x.y; S[4 * c4 + 2] = x.z; S[4 * c4 + 3] = x.w;
            }
        } else {
            // columns 0-63 here, 64-127 from the decay warps through Sbuf (fp32, row t
            // at byte 256 t), which MMA3 does not read before the first put_state
            asm volatile("griddepcontrol.wait;\n" ::: "memory");
            seg_initial_half<0>(S, E, G, bh, P, p, t);
            named_bar(4, 256);
            const float4 *hi = reinterpret_cast<const float4 *>(Sbuf + (size_t)t * 256);
#pragma unroll
            for (int c4 = 0; c4 < 16; ++c4) {
                const float4 x = hi[c4];
                S[64 + 4 * c4] = x.x; S[64 + 4 * c4 + 1] = x.y; S[64 + 4 * c4 + 2] = x.z; S[64 + 4 * c4 + 3] = x.w;
            }
            named_bar(2, 128);  // every row read before put_state overwrites Sbuf
        }
        auto put_state = [&]() {  // bf16 row t of S into the N-major B tile
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
                uint4 v = make_uint4(pack_bf16x2(S[8 * ch], S[8 * ch + 1]), pack_bf16x2(S[8 * ch + 2], S[8 * ch + 3]),
                                     pack_bf16x2(S[8 * ch + 4], S[8 * ch + 5]), pack_bf16x2(S[8 * ch + 6], S[8 * ch + 7]));
                *reinterpret_cast<uint4 *>(Sbuf + tile_chunk(t, ch)) = v;
            }
            fence_proxy_async_smem();
        };
        put_state();
        named_bar(2, 128);
        if (t == 0) mbar_arrive(&sm.s_ready);
        if (p == 0 && P > 1 && YOCO_DCHECK(bh < (size_t)(gridDim.x / P), 0x42)) {
            // the caller's state is in registers now, so the last segment may overwrite
            // it; if that segment has already parked the final state, copy it over
            if (t == 0) {
                __threadfence();
                sm.hand_old = atomicOr(hand + bh, kHandInitRead);
                __threadfence();
            }
            named_bar(2, 128);
            if (sm.hand_old & kHandParked) {
                const float4 *src = reinterpret_cast<const float4 *>(E + (bh * (P + 1) + P) * kD * kD + (size_t)t * kD);
                float4 *dst = reinterpret_cast<float4 *>(state + bh * kD * kD + (size_t)t * kD);
#pragma unroll 8
                for (int c4 = 0; c4 < kD / 4; ++c4) dst[c4] = __ldcg(src + c4);
            }
        }
        float lg_next = (nchunks > 0) ? chunk_log_gate(chunk_start(0), t) : 0.f;
        for (int i = 0; i < nchunks; ++i) {
            // the chunk's decay, computed here too (cheap) so no ring is shared with the decay warps
            float bC;
            (void)group_scan(lg_next, sm.wsum0, lane, warp, 2, bC);
            if (i + 1 < nchunks) lg_next = chunk_log_gate(chunk_start(i + 1), t);
            bool ok = true;
            if (t == 0) {
                ok = mbar_wait(&sm.u_full, i & 1, abort_flag);
                if (!ok) report(err, &sm.abort_flag, 4);
                sm.go0 = ok && !*abort_flag;
            }
            named_bar(2, 128);
            if (!sm.go0) break;
            tc_fence_after();
            const float ebC = __expf(bC);
            const uint64_t ebC2 = f2_pack(ebC, ebC);
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t r[32];
                tmem_ld32(tmem + kColU + lane_base + cb * 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 2)  // S <- e^{b_C} S + U, two columns per packed FMA
                    f2_unpack(f2_fma(ebC2, f2_pack(S[cb * 32 + e], S[cb * 32 + e + 1]),
                                     f2_pack(__uint_as_float(r[e]), __uint_as_float(r[e + 1]))),
                              S[cb * 32 + e], S[cb * 32 + e + 1]);
            }
            tc_fence_before();
            if (i + 1 < nchunks) put_state();  // MMA3 of this chunk is done (u_full)
            named_bar(2, 128);
            if (t == 0) {
                mbar_arrive(&sm.u_free);
                if (i + 1 < nchunks) mbar_arrive(&sm.s_ready);
            }
        }
        named_bar(2, 128);
        if (t == 0) sm.go0 = !*abort_flag;
        named_bar(2, 128);
        if (p == P - 1 && sm.go0) {  // the last segment's end state is the call's final state
            // With P > 1, segment 0 reads the caller's state from `state`: overwrite it
            // only once segment 0 has its copy, else park the final state in slot P for
            // segment 0 to copy (if segment 0 takes its copy in between, write it here too)
            if (P > 1 && t == 0) sm.hand_old = ld_acquire_gpu(hand + bh);
            named_bar(2, 128);
            const bool parked = P > 1 && !(sm.hand_old & kHandInitRead) &&
                                YOCO_DCHECK(bh * (P + 1) + P < (size_t)(gridDim.x / P) * (P + 1), 0x41);
            float *row = parked ? E + (bh * (P + 1) + P) * kD * kD : state + bh * kD * kD;
            for (int pass = 0; pass < 2; ++pass) {
                float4 *dst = reinterpret_cast<float4 *>(row + (size_t)t * kD);
#pragma unroll
                for (int c4 = 0; c4 < kD / 4; ++c4)
                    dst[c4] = make_float4(S[4 * c4], S[4 * c4 + 1], S[4 * c4 + 2], S[4 * c4 + 3]);
                if (!parked || pass == 1) break;
                __threadfence();
                named_bar(2, 128);
                if (t == 0) sm.hand_old = atomicOr(hand + bh, kHandParked);
                named_bar(2, 128);
                if (!(sm.hand_old & kHandInitRead)) break;  // segment 0 will copy the parked state
                row = state + bh * kD * kD;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// Segment end states, read-only over k and v: for segment p of (b, h),
//     E_p = sum_j (prod_{m > j, m in segment} gamma_m) k_j^T v_j,   G_p = sum_j log gamma_j,
// walking the segment's 128-token chunks backwards (the running suffix decay
// weights each token).  The pass streams k and v and does little per byte, so a
// ring slot should be held for as few hand-offs as possible: every token's weight
// is computed from the gate logits before its chunk lands, and the moment it lands
// the eight scale warps rescale K in place (thread = one row-half) and announce it;
// the MMA E^T += V^T (w . K) into TMEM (lane = d_v) then frees the slot.
// The walk stops at the first chunk whose newest token weighs below e^-kDropLog
// (found from the gate logits in a short prologue, 64 chunks per round), and
// G_p is then the decay of the walked chunks, itself below e^-kDropLog.
constexpr int kSegStages = 3;
constexpr int kSegThreads = 320;              // warps 0-7 scale, 8 TMA, 9 MMA
constexpr int kSegScale = 256;
constexpr int kSegScanChunks = 64;            // chunks per round of the walk-length prologue

struct SegSmem {
    uint64_t full[kSegStages], empty[kSegStages], scaled[kSegStages], e_full, decided;
    uint32_t tmem_base;
    int abort_flag;
    int go;
    int nuse;         // chunks the walk takes (decided by the scale warps' prologue)
    float wsum[2][8];
    float csum[64];   // prologue: total log decay of 64 chunks
    float lgc[kSegScanChunks][kC];  // prologue's first round: each token's log gate, walk chunks 0-63
};

constexpr size_t kSegSmemBytes = (size_t)kSegStages * 2 * kTile + sizeof(SegSmem) + 1024;
static_assert(kSegSmemBytes <= kTcSmemBytes, "segment-state ring + control block must fit");

__global__ void __launch_bounds__(kSegThreads, 1)
gret_seg_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const float *__restrict__ logits, float inv_tau, const float *__restrict__ state,
                float *__restrict__ E, float *__restrict__ G, int *__restrict__ hand, int N, int H, int seg_len,
                int P, int *err) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *tiles = smem_raw + pad;
    SegSmem &sm = *reinterpret_cast<SegSmem *>(tiles + (size_t)kSegStages * 2 * kTile);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int p = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int t_begin = p * seg_len;
    const int nch = (min(N, t_begin + seg_len) - t_begin + kC - 1) / kC;
    const size_t bh = (size_t)b * H + h;
    const size_t bhp = bh * P + p;                 // G slot
    const size_t e_slot = bh * (size_t)(P + 1) + p;  // E slot
    [[maybe_unused]] const size_t nbh = (size_t)gridDim.y * gridDim.z;
    const bool slots_ok = YOCO_DCHECK(e_slot < nbh * (P + 1) && p < P - 1, 0x43) && YOCO_DCHECK(bhp < nbh * P, 0x44);
    auto stage_k = [&](int s) { return tiles + (size_t)s * 2 * kTile; };
    auto stage_v = [&](int s) { return tiles + (size_t)s * 2 * kTile + kTile; };
    auto chunk_at = [&](int i) { return t_begin + (nch - 1 - i) * kC; };  // backwards

    if (tid == 0) {
        for (int s = 0; s < kSegStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
            mbar_init(&sm.scaled[s], 1);
        }
        mbar_init(&sm.e_full, 1);
        mbar_init(&sm.decided, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    volatile int *abort_flag = &sm.abort_flag;
    // Programmatic dependent launch: wait for the previous kernel before any global
    // access; clear this call's final-state hand-off word, then let the output grid
    // (which sets and reads it) start.
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    if (p == 0 && tid == 0) {
        *reinterpret_cast<volatile int *>(hand + bh) = 0;
        __threadfence();
    }
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    if (warp == 8) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            const uint64_t pol = l2_policy_evict_first();
            // the first kSegStages chunks are requested before the walk length is known
            // (the newest chunk is always walked); the rest only if the walk takes them
            const int spec = min(nch, kSegStages);
            int lim = spec;
            int i = 0;
            for (;; ++i) {
                if (i == spec) {
                    if (!mbar_wait(&sm.decided, 0, abort_flag)) {
                        report(err, &sm.abort_flag, 35);
                        break;
                    }
                    lim = max(spec, sm.nuse);
                }
                if (i >= lim) break;
                const int s = i % kSegStages;
                if (i >= kSegStages && !mbar_wait(&sm.empty[s], ((i / kSegStages) + 1) & 1, abort_flag)) {
                    report(err, &sm.abort_flag, 31);
                    break;
                }
                const int n0 = chunk_at(i);
                mbar_arrive_expect_tx(&sm.full[s], 2 * kTile);
                for (int half = 0; half < 2; ++half) {
                    tma_load_4d_hint(stage_k(s) + half * kHalf, &tm_k, &sm.full[s], half * 64, h, n0, b, pol);
                    tma_load_4d_hint(stage_v(s) + half * kHalf, &tm_v, &sm.full[s], half * 64, h, n0, b, pol);
                }
            }
            // leave no copy in flight, walked or not (bounded by time only: an abort must still wait)
            volatile int no_abort = 0;
            for (int k = max(0, i - kSegStages); k < i; ++k)
                mbar_wait(&sm.full[k % kSegStages], (k / kSegStages) & 1, &no_abort, 200000000ull);
        }
    } else if (warp == 9) {
        // -------------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t id_kv = idesc_bf16_f32(kD, kD, true, true);  // A = V^T (M-major), B = K'' (N-major)
            bool ok = mbar_wait(&sm.decided, 0, abort_flag);
            const int nuse = ok ? sm.nuse : 0;
            for (int i = 0; i < nuse; ++i) {
                const int s = i % kSegStages;
                if (!(ok = mbar_wait(&sm.scaled[s], (i / kSegStages) & 1, abort_flag))) break;
                tc_fence_after();
                const uint32_t k_a = smem_u32(stage_k(s)), v_a = smem_u32(stage_v(s));
                for (int kk = 0; kk < 8; ++kk)  // E^T += V^T K'', 16 tokens per MMA
                    mma_ss(tmem, smem_desc_sw128(v_a + kk * 2048, kHalf, 1024),
                           smem_desc_sw128(k_a + kk * 2048, kHalf, 1024), id_kv, (i > 0 || kk > 0));
                mma_commit(&sm.empty[s]);
            }
            if (!ok) report(err, &sm.abort_flag, 32);
            mma_commit(&sm.e_full);  // also: nothing of ours runs once it completes
        }
    } else {
        // --------------------------------------------- scale warps (0-7)
        // thread u: row r = u % 128 of the chunk, column half u / 128 of K; warp w scans
        // rows 32 (w % 4) .. 32 (w % 4) + 31
        const int r = tid & (kC - 1), hf = tid >> 7, wr = warp & 3;
        auto log_gate_at = [&](int n0) {
            const int n = n0 + r;
            return (n < N) ? log_gate(logits[((size_t)b * N + n) * H + h], inv_tau) : 0.f;
        };
        // prologue: how many chunks, walking back from the segment end, to take.  Round
        // by round, warp w sums the log decay of chunks c0 + 8w .. c0 + 8w + 7 (32
        // logits in flight per lane); every thread then scans the 64 totals the same
        // way and stops before the first chunk that starts below e^-kDropLog.
        int nuse = nch;
        {
            float run = 0.f;  // log decay of the chunks already taken
            for (int c0 = 0; c0 < nch; c0 += kSegScanChunks) {
                float part[8];
#pragma unroll
                for (int k8 = 0; k8 < 8; ++k8) {
                    part[k8] = 0.f;
                    const int c = c0 + 8 * warp + k8;
                    if (c < nch) {
                        const int n0 = chunk_at(c);
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const int n = n0 + lane + 32 * m;
                            const float lgv =
                                (n < N) ? log_gate(__ldg(logits + ((size_t)b * N + n) * H + h), inv_tau) : 0.f;
                            part[k8] += lgv;
                            if (c0 == 0) sm.lgc[c][lane + 32 * m] = lgv;  // the walk reads them back
                        }
                    }
                }
#pragma unroll
                for (int k8 = 0; k8 < 8; ++k8) {
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) part[k8] += __shfl_xor_sync(0xffffffffu, part[k8], off);
                }
                if (lane < 8) {
                    float pv = part[0];
#pragma unroll
                    for (int k8 = 1; k8 < 8; ++k8) pv = (lane == k8) ? part[k8] : pv;
                    sm.csum[8 * warp + lane] = pv;
                }
                named_bar(1, kSegScale);
                bool stop = false;
                for (int k2 = 0; k2 < kSegScanChunks && c0 + k2 < nch; ++k2) {
                    if (run < -kDropLog) {
                        nuse = c0 + k2;
                        stop = true;
                        break;
                    }
                    run += sm.csum[k2];
                }
                named_bar(1, kSegScale);  // csum is rewritten by the next round
                if (stop) break;
            }
            if (tid == 0) {
                sm.nuse = nuse;
                mbar_arrive(&sm.decided);
            }
        }
        float suffix = 0.f;  // log decay of the chunks after this one
        // walk chunk i's log gate of row r: the prologue kept those of chunks 0-63 (the
        // whole walk unless the gates barely decay); later ones are read as it goes
        auto lg_walk = [&](int i) { return i < kSegScanChunks ? sm.lgc[i][r] : log_gate_at(chunk_at(i)); };
        float lg_next = (nuse > 0) ? lg_walk(0) : 0.f;
        bool alive = true;
        for (int i = 0; i < nuse && alive; ++i) {
            const int s = i % kSegStages;
            float x = lg_next;
            if (i + 1 < nuse) lg_next = lg_walk(i + 1);  // from shared memory, or in flight during this chunk
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            if (lane == 31) sm.wsum[i & 1][warp] = x;
            named_bar(1, kSegScale);
            float pre = 0.f, bC = 0.f;
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
                const float t = sm.wsum[i & 1][w4];
                bC += t;
                if (w4 < wr) pre += t;
            }
            // weight of token r: decay from r (exclusive) to the segment end
            const float w = __expf(suffix + (bC - (x + pre)));
            suffix += bC;
            if (tid == 0) {
                const bool ok = mbar_wait(&sm.full[s], (i / kSegStages) & 1, abort_flag);
                if (!ok) report(err, &sm.abort_flag, 33);
                sm.go = ok && !*abort_flag;
            }
            named_bar(1, kSegScale);
            if (!sm.go) {
                alive = false;
                break;
            }
            {  // row r, columns 64 hf .. 64 hf + 63 of K, in place (128-byte swizzle)
                const __nv_bfloat162 w2 = __float2bfloat162_rn(w);
                uint8_t *row = stage_k(s) + hf * kHalf + r * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 *q = reinterpret_cast<uint4 *>(row + ((c ^ (r & 7)) * 16));
                    *q = scale_bf16x8(*q, w2);
                }
            }
            fence_proxy_async_smem();
            named_bar(1, kSegScale);
            if (tid == 0) mbar_arrive(&sm.scaled[s]);
        }
        if (tid == 0 && slots_ok) G[bhp] = suffix;
        if (p == 0 && tid < kD) {  // keep the caller's initial state: the OUTPUT pass overwrites `state`
            const float4 *src = reinterpret_cast<const float4 *>(state + bh * kD * kD + (size_t)tid * kD);
            float4 *dst = reinterpret_cast<float4 *>(E + (bh * (P + 1) + P - 1) * kD * kD + (size_t)tid * kD);
#pragma unroll 4
            for (int c4 = 0; c4 < kD / 4; ++c4) dst[c4] = src[c4];
        }
        if (tid == 0) {
            const bool ok = mbar_wait(&sm.e_full, 0, abort_flag, 4000000000ull);
            if (!ok) report(err, &sm.abort_flag, 34);
            sm.go = ok && !*abort_flag;
        }
        named_bar(1, kSegScale);
        if (sm.go && alive && slots_ok && tid < kD) {
            // E^T row tid (lane = d_v column tid) -> E[d_k][d_v]
            tc_fence_after();
            const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + cb * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) E[e_slot * kD * kD + (size_t)(cb * 32 + e) * kD + tid] = __uint_as_float(v[e]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 128);
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

// Segments per head: the output kernel runs one CTA per SM (its shared memory), so
// about one CTA per SM of the device over the B*H heads.
static int tc_segments(int B, int N, int H) {
    const int chunks = (N + kC - 1) / kC;
    const int forced = (int)test_hook_value(kHookGretSegments);  // 0: off (tests and measurements)
    int P = forced > 0 ? forced : device_sm_count() / (B * H);
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
    // per (b, h): P + 1 states (end states of segments 0 .. P-2, the caller's initial
    // state, the parked final state), P segment decays and the hand-off word
    if (P > 1) ws += ((size_t)B * H * (P + 1) * kD * kD + (size_t)B * H * P) * sizeof(float) + (size_t)B * H * sizeof(int);
    return ws;
}

// The chunkwise prefill on the tensor cores.  gn == nullptr: o = the retention
// output; else o = Eq. 7's z = swish(gate) (.) GroupNorm_h(retention output).
cudaError_t gret_prefill_tc(const GretArgs &a, const GnArgs *gn, void *ws, cudaStream_t st) {
    CUtensorMap mq, mk, mv, mo, mg;
    if (!make_map(&mq, a.q, a.B, a.N, a.H) || !make_map(&mk, a.k, a.B, a.N, a.H) || !make_map(&mv, a.v, a.B, a.N, a.H) ||
        !make_map(&mo, a.o, a.B, a.N, a.H))
        return cudaErrorInvalidValue;
    // the gate of Eq. 7 (same layout as q; without it the map is not used)
    if (gn) {
        if (!make_map(&mg, gn->gate, a.B, a.N, a.H)) return cudaErrorInvalidValue;
    } else {
        mg = mq;
    }
    int P = tc_segments(a.B, a.N, a.H);
    const int seg_len = tc_seg_len(a.N, P);
    P = (a.N + seg_len - 1) / seg_len;
    int *err = (int *)ws;
    float *E = (float *)((char *)ws + 256);
    float *G = E + (size_t)a.B * a.H * (P + 1) * kD * kD;
    int *hand = reinterpret_cast<int *>(G + (size_t)a.B * a.H * P);
    const float inv_tau = 1.0f / a.tau;
    auto out_kernel = gn ? gret_tc_kernel<true> : gret_tc_kernel<false>;
    const bf16_t *gate = gn ? (const bf16_t *)gn->gate : nullptr;
    const float *gn_w = gn ? gn->w : nullptr, *gn_b = gn ? gn->b : nullptr;
    const float gn_eps = gn ? gn->eps : 0.f;
    cudaError_t e;
    e = cudaFuncSetAttribute(out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gret_seg_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSegSmemBytes);
    if (e != cudaSuccess) return e;
    if (P == 1) {
        count_launches(1);
        out_kernel<<<dim3(a.B * a.H), kTcThreads, kTcSmemBytes, st>>>(
            mq, mk, mv, mo, mg, a.logits, inv_tau, a.state, E, G, nullptr, a.N, a.H, seg_len, 1, err, (uint64_t)0, gate,
            gn_w, gn_b, gn_eps);
        return cudaGetLastError();
    }
    // end states of segments 0 .. P-2 (the last segment's is computed by the OUTPUT pass)
    count_launches(2);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // segment states: the prologue overlaps the previous kernel's tail; it waits for it
    // before reading anything
    cfg.gridDim = dim3(P - 1, a.H, a.B);
    cfg.blockDim = dim3(kSegThreads);
    cfg.dynamicSmemBytes = kSegSmemBytes;
    e = cudaLaunchKernelEx(&cfg, gret_seg_kernel, mk, mv, a.logits, inv_tau, (const float *)a.state, E, G, hand,
                           a.N, a.H, seg_len, P, err);
    if (e != cudaSuccess) return e;
    // the output grid starts on the SMs the segment-state grid leaves free: its segment-0 CTAs (first in
    // the grid) run the whole segment meanwhile; the others begin loading and wait
    // for the segment states before touching E, G and `state`
    cfg.gridDim = dim3(P * a.B * a.H);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = kTcSmemBytes;
    return cudaLaunchKernelEx(&cfg, out_kernel, mq, mk, mv, mo, mg, a.logits, inv_tau, a.state, E, G, hand, a.N, a.H,
                              seg_len, P, err, (uint64_t)test_hook_value(kHookGretSeg0DelayNs), gate, gn_w, gn_b,
                              gn_eps);
}

}  // namespace yoco_host

YOCO_DEBUG_TU(gret_tc)
