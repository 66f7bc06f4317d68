// kernels.h -- host-side launchers behind the C ABI (internal to libyoco).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "yoco.h"

namespace yoco_host {

// Streaming multiprocessors of the current device (queried once per device).  Grids
// are sized from it; kDefaultSmCount (a GB300's 152) stands in only where no device
// can be queried (workspace-size queries on a machine without a GPU).
constexpr int kDefaultSmCount = 152;
int device_sm_count();

// Test hooks (yoco_test_hook): process-wide values that tests set to reach paths
// ordinary inputs cannot force; all are 0 (off) unless a test sets them.
enum { kHookFailNextCalls = 1, kHookGretSeg0DelayNs = 2, kHookGretSegments = 3, kHookCount = 4 };
int64_t test_hook_value(int hook);
// true (and the call must return YOCO_ERR_CUDA before launching anything) while an
// injected launch failure is pending; consumes one
bool take_injected_failure();

struct GretArgs {
    const void *q, *k, *v;
    const float *logits;
    float tau;
    void *o;
    float *state;
    int B, N, H, dk, dv;
    yoco_dtype in_dt;
};

// gret_simt.cu
size_t gret_simt_smem_bytes(int dk);
size_t gret_simt_workspace(int B, int N, int H, int dk, int dv);
cudaError_t gret_prefill_simt(const GretArgs &a, void *ws, cudaStream_t st);
// segment join shared by both paths: E[bh][p] (zero-start end states) -> initial states
cudaError_t gret_scan_launch(float *E, const float *G, float *state, int BH, int P, int DD, cudaStream_t st);
cudaError_t gret_decode(const void *q, const void *k, const void *v, const float *logits, float tau,
                        float *state, void *o, int B, int H, int dk, int dv, yoco_dtype dt, cudaStream_t st);
// the recurrent step followed by GroupNorm_h + swish gate (one cluster per head)
cudaError_t gret_decode_gn(const void *q, const void *k, const void *v, const float *logits, float tau,
                           float *state, const void *gate, const float *gn_w, const float *gn_b, float eps, void *z,
                           int B, int H, int dk, int dv, yoco_dtype dt, cudaStream_t st);

// gret_tc.cu (bf16, d = 128, tensor cores)
struct GnArgs {  // Eq. 7 output: z = swish(gate) (.) GroupNorm_h(o)
    const void *gate;
    const float *w, *b;  // per-channel affine [H * d] or NULL
    float eps;
};
bool gret_tc_eligible(int B, int N, int H, int dk, int dv, yoco_dtype dt);
size_t gret_tc_workspace(int B, int N, int H, int dk, int dv);
cudaError_t gret_prefill_tc(const GretArgs &a, const GnArgs *gn, void *ws, cudaStream_t st);

// kv_proj.cu
struct KvProjArgs {
    const void *M, *rms_w, *Wk, *Wv;
    float eps;
    int B, T, dm, Hkv, d;
    int64_t cap, len;
    void *kc, *vc;
    int32_t *len_dev;
    yoco_dtype dt;
    float rope_base;  // 0: K^ is not rotated
};
size_t kv_proj_workspace(int B, int T, int dm, int Hkv, int d, yoco_dtype dt, float rope_base);
cudaError_t kv_project_append(const KvProjArgs &a, void *ws, cudaStream_t st);
// kv_proj_tc.cu: bf16, no gain, Hkv*d % 256 == 0, >= 128 rows
bool kv_proj_tc_eligible(const KvProjArgs &a);
cudaError_t kv_project_append_tc(const KvProjArgs &a, const float *rrow, const float2 *rope_cs, int *err,
                                 cudaStream_t st);

// attn.cu
struct AttnArgs {
    const void *Q;
    void *O;
    const void *kc, *vc;
    int B, T, Hq, Hkv, d;
    int64_t cap, p0;  // row t sits at position p0 + t
    float scale;
    yoco_dtype dt;
    float rope_base;  // 0: queries are not rotated
};
// resident CTAs per SM of the decode kernel that will run: 1 for the tensor-core
// kernel (bf16, d = 128, <= 16 query heads per kv head), 3 for the CUDA-core one
int attn_ctas_per_sm(yoco_dtype dt, int d, int group);
int attn_auto_splits(int B, int Hkv, int64_t keys, int ctas_per_sm);
size_t attn_workspace(int B, int Hq, int T, int d, int splits);
cudaError_t attn_run(const AttnArgs &a, int splits, void *ws, cudaStream_t st);
// attn_tc.cu: bf16, d = 128, <= 16 query vectors per CTA
bool attn_tc_eligible(const AttnArgs &a, int nq);
cudaError_t attn_tc_launch(const AttnArgs &a, int RB, int nq, int64_t kps, int splits, void *part, int *err,
                           cudaStream_t st);

// attn_fa.cu: many query rows (prefill), bf16, d = 128; window > 0 adds the sliding-window mask
bool attn_fa_eligible(const AttnArgs &a);
cudaError_t attn_fa_launch(const AttnArgs &a, int64_t window, int *err, cudaStream_t st);
// sliding-window self-attention over token-major q [B,N,Hq,128], k, v [B,N,Hkv,128] (bf16)
cudaError_t swa_fa_launch(const void *q, const void *k, const void *v, void *o, int B, int N, int Hq, int Hkv,
                          int64_t window, float scale, int *err, cudaStream_t st);
// swa.cu: copy tokens [tok0, tok0 + n) of k, v [B, N, Hkv, d] to ring slots (pos0 + i) % window
cudaError_t swa_ring_write(const void *k, const void *v, void *rk, void *rv, int B, int N, int Hkv, int d,
                           int window, int64_t tok0, int n, int64_t pos0, yoco_dtype dt, cudaStream_t st);

// gn_gate.cu: z = swish(gate) * GroupNorm_h(o) over rows of d (one group per head)
cudaError_t group_norm_gate(const void *o, const void *gate, const float *w, const float *b, float eps, void *z,
                            int64_t rows, int H, int d, yoco_dtype dt, cudaStream_t st);

// rope.cu: rotary encoding of token-major x [B, N, H, d] in place, row n at position pos0 + n
cudaError_t rope_apply(void *x, int B, int N, int H, int d, int64_t pos0, float base, yoco_dtype dt, cudaStream_t st);
// (cos, sin) of (pos0 + t) theta_i into tab [T][d/2] (float2)
cudaError_t rope_table(float2 *tab, int64_t pos0, int T, int d, float base, cudaStream_t st);

// qkvg_tc.cu: [q | k | v | logits] = X [W_Q | W_K | W_V | W_gamma], bf16, tensor cores
cudaError_t qkvg_project(const void *X, const void *W, int B, int N, int dm, int H, int d, void *q, void *k, void *v,
                         float *logits, const float2 *rope_cs, int *err, cudaStream_t st);

// debug builds: each kernel file's debug word (see YOCO_DEBUG_TU in common.cuh)
#define YOCO_DEBUG_TUS(X) X(attn) X(attn_fa) X(attn_tc) X(gn_gate) X(gret_simt) X(gret_tc) X(kv_proj) \
    X(kv_proj_tc) X(qkvg_tc) X(rope) X(swa)
#define YOCO_DECLARE_DEBUG_WORD(tu) cudaError_t debug_word_##tu(unsigned *w, int clear);
YOCO_DEBUG_TUS(YOCO_DECLARE_DEBUG_WORD)

// selftest.cu
cudaError_t selftest_wait(void *ws, uint64_t limit_ns, cudaStream_t st);
cudaError_t selftest_occupy(int ctas, uint64_t ns, cudaStream_t st);

}  // namespace yoco_host
