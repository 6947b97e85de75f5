// MiniMax tensor-parallel QK-RMSNorm with the R shards resident on one GPU,
// as one fused kernel (vLLM rms_norm_tp: `_minimax_qk_var_kernel`, the
// all-reduce of the [T, 2] fp32 variance, `_minimax_rms_apply_kernel`).  With
// no k segment (K == 0, KC == 0) the same kernel is the single-matrix sharded
// RMSNorm of tokenspeed trtllm.py `minimax_allreduce_rms`.
//
// One warp per (token, shard): the warp reads the shard's q (Q values) and k
// (K values) of the token once into registers (128-bit loads, lane l owns
// chunks l, l+32, ...), reduces the per-shard means of squares with shuffles,
// and parks them in shared memory.  After one barrier every warp of the token
// sums the R shard means in ascending shard order (the all-reduce, here a
// local fp32 sum), takes rsqrt(V/R + eps) and writes its block of q_out /
// k_out from the registers.  Several tokens share a CTA when R is small.
#include "device_util.cuh"
#include "launch.h"

namespace tsfn {

namespace {

constexpr int kMaxThreads = 512;

template <int QC, int KC>
__global__ void __launch_bounds__(kMaxThreads) qk_norm_kernel(const __grid_constant__ QKArgs a, int tpc)
{
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tl = warp / a.R;
    const int r = warp - tl * a.R;
    const int64_t t = (int64_t)blockIdx.x * tpc + tl;
    const bool live = t < a.T;
    const int qn = a.Q >> 3, kn = a.K >> 3;

    __shared__ float mq[kMaxThreads / 32], mk[kMaxThreads / 32];

    pdl_wait();

    const uint16_t *base = a.shards[r] + t * a.row_stride;
    uint4 qv[QC], kv[KC > 0 ? KC : 1];
#pragma unroll
    for (int i = 0; i < QC; ++i) {
        const int c = lane + 32 * i;
        if (live && c < qn)
            qv[i] = ld_stream(base + (int64_t)c * 8);
    }
#pragma unroll
    for (int i = 0; i < KC; ++i) {
        const int c = lane + 32 * i;
        if (live && c < kn)
            kv[i] = ld_stream(base + a.Q + (int64_t)c * 8);
    }
    float sq = 0.0f, sk = 0.0f;
#pragma unroll
    for (int i = 0; i < QC; ++i) {
        const int c = lane + 32 * i;
        if (live && c < qn) {
            float f[8];
            unpack8(qv[i], f);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                sq = fmaf(f[e], f[e], sq);
        }
    }
#pragma unroll
    for (int i = 0; i < KC; ++i) {
        const int c = lane + 32 * i;
        if (live && c < kn) {
            float f[8];
            unpack8(kv[i], f);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                sk = fmaf(f[e], f[e], sk);
        }
    }
    pdl_launch_dependents();
    sq = warp_sum(sq);
    if (KC > 0)
        sk = warp_sum(sk);
    if (lane == 0) {
        mq[warp] = __fdiv_rn(sq, (float)a.Q);
        if (KC > 0)
            mk[warp] = __fdiv_rn(sk, (float)a.K);
    }
    __syncthreads();
    if (!live)
        return;

    float Vq = 0.0f, Vk = 0.0f;
    for (int s = 0; s < a.R; ++s) {
        Vq = __fadd_rn(Vq, mq[tl * a.R + s]);
        if (KC > 0)
            Vk = __fadd_rn(Vk, mk[tl * a.R + s]);
    }
    const float iq = rsqrtf(__fadd_rn(__fdiv_rn(Vq, (float)a.R), a.eps));
    const float ik = KC > 0 ? rsqrtf(__fadd_rn(__fdiv_rn(Vk, (float)a.R), a.eps)) : 0.0f;

    const uint16_t *wq = a.q_weight + (int64_t)r * a.Q;
    uint16_t *qo = a.q_out + t * a.ldq + (int64_t)r * a.Q;
#pragma unroll
    for (int i = 0; i < QC; ++i) {
        const int c = lane + 32 * i;
        if (c < qn) {
            float f[8], w[8], y[8];
            unpack8(qv[i], f);
            unpack8(ld_keep(wq + (int64_t)c * 8), w);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                y[e] = __fmul_rn(__fmul_rn(f[e], iq), w[e]);
            st_v4(qo + (int64_t)c * 8, pack8(y));
        }
    }
    if constexpr (KC == 0)
        return;
    const uint16_t *wk = a.k_weight + (int64_t)r * a.K;
    uint16_t *ko = a.k_out + t * a.ldk + (int64_t)r * a.K;
#pragma unroll
    for (int i = 0; i < KC; ++i) {
        const int c = lane + 32 * i;
        if (c < kn) {
            float f[8], w[8], y[8];
            unpack8(kv[i], f);
            unpack8(ld_keep(wk + (int64_t)c * 8), w);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                y[e] = __fmul_rn(__fmul_rn(f[e], ik), w[e]);
            st_v4(ko + (int64_t)c * 8, pack8(y));
        }
    }
}

template <int QC>
cudaError_t launch_qc(const QKArgs &a, int kc, int tpc, int64_t grid, int nthr, bool pdl, cudaStream_t s)
{
    const dim3 g((unsigned)grid), b((unsigned)nthr);
    switch (kc) {
    case 0: return launch_kernel(qk_norm_kernel<QC, 0>, g, b, 0, s, pdl, a, tpc);
    case 1: return launch_kernel(qk_norm_kernel<QC, 1>, g, b, 0, s, pdl, a, tpc);
    case 2: return launch_kernel(qk_norm_kernel<QC, 2>, g, b, 0, s, pdl, a, tpc);
    default: return launch_kernel(qk_norm_kernel<QC, 4>, g, b, 0, s, pdl, a, tpc);
    }
}

// Smallest power of two >= the number of 8-element chunks each lane owns.
int chunks_bucket(int elems)
{
    if (elems == 0)
        return 0;
    const int per_lane = (elems / 8 + 31) / 32;
    int b = 1;
    while (b < per_lane)
        b <<= 1;
    return b;
}

}  // namespace

cudaError_t launch_qk(const QKArgs &a, bool pdl, cudaStream_t stream)
{
    const int qc = chunks_bucket(a.Q);      // 1..16
    const int kc = chunks_bucket(a.K);      // 0..4
    const int tpc = a.R >= 8 ? 1 : 8 / a.R;  // tokens per CTA
    const int nthr = tpc * a.R * 32;
    const int64_t grid = (a.T + tpc - 1) / tpc;
    switch (qc) {
    case 1: return launch_qc<1>(a, kc, tpc, grid, nthr, pdl, stream);
    case 2: return launch_qc<2>(a, kc, tpc, grid, nthr, pdl, stream);
    case 4: return launch_qc<4>(a, kc, tpc, grid, nthr, pdl, stream);
    case 8: return launch_qc<8>(a, kc, tpc, grid, nthr, pdl, stream);
    default: return launch_qc<16>(a, kc, tpc, grid, nthr, pdl, stream);
    }
}

}  // namespace tsfn
