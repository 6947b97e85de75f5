// MiniMax tensor-parallel QK-RMSNorm with the R shards resident on one GPU,
// as one fused kernel (vLLM rms_norm_tp: `_minimax_qk_var_kernel`, the
// all-reduce of the [T, 2] fp32 variance, `_minimax_rms_apply_kernel`).  With
// no k segment (K == 0, KC == 0) the same kernel is the single-matrix sharded
// RMSNorm of tokenspeed trtllm.py `minimax_allreduce_rms`.
//
// One warp per (token, shard), or per two consecutive tokens of a shard when
// its row is narrow: the warp reads the shard's q (Q values) and k (K values)
// of the token once into registers (128-bit loads, lane l owns chunks l,
// l+32, ...), reduces the per-shard means of squares with shuffles,
// and parks them in shared memory.  After one barrier every warp of the token
// sums the R shard means in ascending shard order (the all-reduce, here a
// local fp32 sum), takes rsqrt(V/R + eps) and writes its block of q_out /
// k_out from the registers.  Several tokens share a CTA when R is small.
#include <initializer_list>

#include "device_util.cuh"
#include "launch.h"

namespace tsfn {

namespace {

constexpr int kMaxThreads = 512;

// RN(s / n): a multiply by the exact reciprocal when n is a power of two (the
// same correctly rounded quotient), else an IEEE divide.  The choice is the
// same for the whole launch.
__device__ __forceinline__ float mean_of(float s, int n, float inv_pow2)
{
    return inv_pow2 != 0.0f ? __fmul_rn(s, inv_pow2) : __fdiv_rn(s, (float)n);
}

// TPW consecutive tokens per warp (same shard): 2 where a shard row is at
// most 3 chunks per lane, so that each lane keeps as many 16-byte loads in
// flight as a wider row gives it.  At most 4 q chunks per lane: 64 registers,
// so that two 512-thread CTAs fit an SM.
template <int QC, int KC, int TPW>
__global__ void __launch_bounds__(kMaxThreads, (QC <= 4 ? 2 : 1)) qk_norm_kernel(const __grid_constant__ QKArgs a, int tpc)
{
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tl = (int)div_by((uint32_t)warp, a.div_r);
    const int r = warp - tl * a.R;
    const int64_t t0 = ((int64_t)blockIdx.x * tpc + tl) * TPW;
    const int qn = a.Q >> 3, kn = a.K >> 3;

    __shared__ float mq[kMaxThreads / 32][TPW], mk[kMaxThreads / 32][TPW];

    pdl_wait();

    // q|k of this shard for the tokens a warp one wave later will take: into
    // L2 with one bulk request each, so DRAM stays busy during this warp's
    // reduction and barrier (QK R=8 T=32768: 177.1 us against 179.7 without;
    // single-matrix W=768: 119.9 against 121.4)
    if (lane == 0 && a.prefetch_tokens > 0) {
#pragma unroll
        for (int j = 0; j < TPW; ++j) {
            const int64_t tt = t0 + j + a.prefetch_tokens;
            if (tt < a.T)
                prefetch_l2(a.shards[r] + tt * a.row_stride, (uint32_t)((a.Q + a.K) * 2));
        }
    }

    uint4 qv[TPW][QC], kv[TPW][KC > 0 ? KC : 1];
#pragma unroll
    for (int j = 0; j < TPW; ++j) {
        const bool live = t0 + j < a.T;
        const uint16_t *base = a.shards[r] + (t0 + j) * a.row_stride;
#pragma unroll
        for (int i = 0; i < QC; ++i) {
            const int c = lane + 32 * i;
            if (live && c < qn)
                qv[j][i] = ld_stream(base + (int64_t)c * 8);
        }
#pragma unroll
        for (int i = 0; i < KC; ++i) {
            const int c = lane + 32 * i;
            if (live && c < kn)
                kv[j][i] = ld_stream(base + a.Q + (int64_t)c * 8);
        }
    }
    float sq[TPW], sk[TPW];
#pragma unroll
    for (int j = 0; j < TPW; ++j) {
        const bool live = t0 + j < a.T;
        sq[j] = 0.0f;
        sk[j] = 0.0f;
#pragma unroll
        for (int i = 0; i < QC; ++i) {
            const int c = lane + 32 * i;
            if (live && c < qn)
                sq[j] = sumsq_bf16x8(qv[j][i], sq[j]);
        }
#pragma unroll
        for (int i = 0; i < KC; ++i) {
            const int c = lane + 32 * i;
            if (live && c < kn)
                sk[j] = sumsq_bf16x8(kv[j][i], sk[j]);
        }
    }
    pdl_launch_dependents();
#pragma unroll
    for (int j = 0; j < TPW; ++j) {
        sq[j] = warp_sum(sq[j]);
        if (KC > 0)
            sk[j] = warp_sum(sk[j]);
        if (lane == 0) {
            mq[warp][j] = mean_of(sq[j], a.Q, a.inv_q);
            if (KC > 0)
                mk[warp][j] = mean_of(sk[j], a.K, a.inv_k);
        }
    }
    // One token per warp and at most 5 chunks per lane: the shard's weights
    // are requested before the barrier instead of one chunk at a time behind
    // the previous chunk's stores (QK R=8 T=32768 Q=1024 K=128: 175.4 us
    // against 176.5).
    constexpr bool kEarlyW = TPW == 1 && QC + KC <= 5;
    uint4 wqv[QC], wkv[KC > 0 ? KC : 1];
    if constexpr (kEarlyW) {
#pragma unroll
        for (int i = 0; i < QC; ++i) {
            const int c = lane + 32 * i;
            if (c < qn)
                wqv[i] = ld_keep(a.q_weight + (int64_t)r * a.Q + (int64_t)c * 8);
        }
#pragma unroll
        for (int i = 0; i < KC; ++i) {
            const int c = lane + 32 * i;
            if (c < kn)
                wkv[i] = ld_keep(a.k_weight + (int64_t)r * a.K + (int64_t)c * 8);
        }
    }
    __syncthreads();

#pragma unroll
    for (int j = 0; j < TPW; ++j) {
        const int64_t t = t0 + j;
        if (t >= a.T)
            break;
        float Vq = 0.0f, Vk = 0.0f;
        for (int s = 0; s < a.R; ++s) {
            Vq = __fadd_rn(Vq, mq[tl * a.R + s][j]);
            if (KC > 0)
                Vk = __fadd_rn(Vk, mk[tl * a.R + s][j]);
        }
        const float iq = rsqrtf(__fadd_rn(mean_of(Vq, a.R, a.inv_r), a.eps));
        const float ik = KC > 0 ? rsqrtf(__fadd_rn(mean_of(Vk, a.R, a.inv_r), a.eps)) : 0.0f;

        const uint16_t *wq = a.q_weight + (int64_t)r * a.Q;
        uint16_t *qo = a.q_out + t * a.ldq + (int64_t)r * a.Q;
#pragma unroll
        for (int i = 0; i < QC; ++i) {
            const int c = lane + 32 * i;
            if (c < qn) {
                float f[8], w[8], y[8];
                unpack8(qv[j][i], f);
                if constexpr (kEarlyW)
                    unpack8(wqv[i], w);
                else
                    unpack8(ld_keep(wq + (int64_t)c * 8), w);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    y[e] = __fmul_rn(__fmul_rn(f[e], iq), w[e]);
                st_v4(qo + (int64_t)c * 8, pack8(y));
            }
        }
        if constexpr (KC > 0) {
            const uint16_t *wk = a.k_weight + (int64_t)r * a.K;
            uint16_t *ko = a.k_out + t * a.ldk + (int64_t)r * a.K;
#pragma unroll
            for (int i = 0; i < KC; ++i) {
                const int c = lane + 32 * i;
                if (c < kn) {
                    float f[8], w[8], y[8];
                    unpack8(kv[j][i], f);
                    if constexpr (kEarlyW)
                        unpack8(wkv[i], w);
                    else
                        unpack8(ld_keep(wk + (int64_t)c * 8), w);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        y[e] = __fmul_rn(__fmul_rn(f[e], ik), w[e]);
                    st_v4(ko + (int64_t)c * 8, pack8(y));
                }
            }
        }
    }
}

template <int QC, int KC>
cudaError_t launch_qkc(const QKArgs &a, int tpc, int nthr, bool pdl, cudaStream_t s)
{
    constexpr int tpw = QC + KC <= 3 ? 2 : 1;  // tokens per warp
    const int64_t per_cta = (int64_t)tpc * tpw;
    const dim3 g((unsigned)((a.T + per_cta - 1) / per_cta)), b((unsigned)nthr);
    // one wave of tokens ahead: SMs x resident CTAs per SM x tokens per CTA
    QKArgs c = a;
    c.prefetch_tokens = 0;
    int dev = 0;
    const int sms = current_device_sms(&dev);
    if (sms > 0) {
        // resident CTAs per SM of this instance at nthr (a multiple of 32, at
        // most 16 warps), from the occupancy calculator once per device
        static std::atomic<int> occupancy[kMaxCachedDevices][17];  // per_sm + 1; 0: not computed
        const int w = nthr >> 5;
        const bool cached = dev < kMaxCachedDevices && w <= 16;
        int per_sm = cached ? occupancy[dev][w].load(std::memory_order_relaxed) - 1 : -1;
        if (per_sm < 0) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, qk_norm_kernel<QC, KC, tpw>, nthr, 0) !=
                cudaSuccess)
                per_sm = 0;
            else if (cached)
                occupancy[dev][w].store(per_sm + 1, std::memory_order_relaxed);
        }
        c.prefetch_tokens = (int64_t)sms * per_sm * per_cta;
    }
    return launch_kernel(qk_norm_kernel<QC, KC, tpw>, g, b, 0, s, pdl, c, tpc);
}

template <int QC>
cudaError_t launch_qc(const QKArgs &a, int kc, int tpc, int nthr, bool pdl, cudaStream_t s)
{
    switch (kc) {
    case 0: return launch_qkc<QC, 0>(a, tpc, nthr, pdl, s);
    case 1: return launch_qkc<QC, 1>(a, tpc, nthr, pdl, s);
    case 2: return launch_qkc<QC, 2>(a, tpc, nthr, pdl, s);
    default: return launch_qkc<QC, 4>(a, tpc, nthr, pdl, s);
    }
}

// Number of 8-element chunks each lane owns, rounded up to an instantiated
// count (q: 1, 2, 3, 4, 6, 8, 12, 16; k: 1, 2, 4), so that no unrolled
// iteration is dead for every lane (W = 768 is 3 chunks per lane).
int chunks_per_lane(int elems) { return (elems / 8 + 31) / 32; }

int q_bucket(int elems)
{
    const int n = chunks_per_lane(elems);
    for (int b : {1, 2, 3, 4, 6, 8, 12})
        if (n <= b)
            return b;
    return 16;
}

int k_bucket(int elems)
{
    const int n = chunks_per_lane(elems);
    return n == 0 ? 0 : n <= 1 ? 1 : n <= 2 ? 2 : 4;
}

}  // namespace

cudaError_t launch_qk(const QKArgs &a, bool pdl, cudaStream_t stream)
{
    const int qc = q_bucket(a.Q);           // 1..16
    const int kc = k_bucket(a.K);           // 0..4
    const int tpc = a.R >= 8 ? 1 : 8 / a.R;  // tokens per CTA
    const int nthr = tpc * a.R * 32;
    switch (qc) {
    case 1: return launch_qc<1>(a, kc, tpc, nthr, pdl, stream);
    case 2: return launch_qc<2>(a, kc, tpc, nthr, pdl, stream);
    case 3: return launch_qc<3>(a, kc, tpc, nthr, pdl, stream);
    case 4: return launch_qc<4>(a, kc, tpc, nthr, pdl, stream);
    case 6: return launch_qc<6>(a, kc, tpc, nthr, pdl, stream);
    case 8: return launch_qc<8>(a, kc, tpc, nthr, pdl, stream);
    case 12: return launch_qc<12>(a, kc, tpc, nthr, pdl, stream);
    default: return launch_qc<16>(a, kc, tpc, nthr, pdl, stream);
    }
}

}  // namespace tsfn
