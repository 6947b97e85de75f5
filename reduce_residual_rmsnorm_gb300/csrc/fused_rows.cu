// Fused reduce -> residual -> RMSNorm -> {bf16 | FP8 | NVFP4} epilogue,
// one CTA per token row.
//
// The math is the one of tokenspeed triton.py `amd_allreduce_residual_rmsnorm_kernel`
// (and `amd_all_reduce_kernel` for kAllReduce): the R partials are widened to
// fp32 and added in ascending order into an accumulator that starts at +0,
// the optional add_in of the reduce-scatter "Add" patterns (trtllm.py
// `ReduceScatterFusionPattern`) and then the residual are added in fp32, the
// row's mean of squares of that unrounded fp32 x gives s = rsqrt(mean + eps),
// and n = bf16((x * s) * gamma).  The quantisers of trtllm.py
// `AllReduceFusionPattern` then read n:
//   FP8 per tensor   code = e4m3(n * sigma)
//   FP8 1x128 block  s_g = amax/448, code = e4m3(n / s_g)  (0 if s_g == 0)
//   NVFP4 16-block   SF = e4m3(g * (amax/6)), code = e2m1(n * (g / value(SF)))
//
// Layout of the work: row t is H/8 chunks of 8 bf16 (16 bytes).  Thread i of
// the CTA owns chunks i, i + blockDim, ... (V of them), so a warp covers 32
// consecutive chunks = 512 contiguous bytes of every tensor; a 1x128 FP8 group
// is 16 consecutive lanes and an NVFP4 block 2 consecutive lanes, so the group
// maxima are warp shuffles.  x stays in registers between the two phases; the
// only shared memory is the per-warp partial sums of x^2.
#include "device_util.cuh"
#include "launch.h"
#include "sf_layout.cuh"

namespace tsfn {

namespace {

constexpr int kMaxThreads = 512;
constexpr int kMaxThreadsPaired = 1024;  // a layout of up to 512 threads spread over pairs (PAIRED)

// Register cap per instance (unpaired CTAs have at most kMaxThreads = 512
// threads, so every cap <= 128 keeps a full CTA launchable; paired CTAs of up
// to 1024 threads exist only for at most 8 partials and 2 chunks per thread,
// whose cap of 64 fills the 65536 registers exactly): at most 8 partials and
// 2 chunks per thread must leave room for two 512-thread CTAs per SM (64
// registers).  The tests check that no instance spills.
template <int RB, int V>
constexpr int reg_cap()
{
    return (RB <= 8 && V <= 2) ? 64 : 128;
}

// Chunks whose loads a thread issues together before consuming them.  With at
// most 4 partials and 2 chunks per thread, both chunks' R+1 loads fit in the
// 64 registers, which keeps twice the bytes in flight per thread (R=4 T=8192
// H=7168: 117.0 us against 125.3 us one chunk at a time, at 48 registers and
// one more CTA per SM); with 8 partials the 18 loads of two chunks would not.
template <int RB, int V>
constexpr int load_group()
{
    return (RB <= 4 && V <= 2) ? V : 1;
}

// PAIRED: the layout of 2V chunks per thread on nthr/2 threads, spread over
// nthr threads of V chunks.  Thread i holds the first V chunks of a 2V-chunk
// thread and thread i + nthr/2 the last V; the first passes its running sum
// of squares to the second, which continues the same chain, so every value
// and every rounding is the one of the 2V-chunk layout: a row's outputs do
// not depend on T.
//
// WAIT, the place of the dependency wait of a launch with programmatic
// dependent launch:
//   kWaitFirst  before the first memory access (TS_FLAG_PDL alone);
//   kEarlyRead  after the first chunk group's loads are issued, so that they
//               overlap the previous kernel's last CTAs; nothing is written
//               before the wait (TS_FLAG_PDL_EARLY_READ: the previous kernel
//               writes none of this call's inputs);
//   kWaitLast   just before each thread exits, after all of its work, so the
//               whole call can run beside the previous kernel and still
//               completes after it (TS_FLAG_PDL_INDEPENDENT: the previous
//               kernel writes none of this call's inputs and neither reads nor
//               writes its outputs).
enum : int { kWaitFirst = 0, kEarlyRead = 1, kWaitLast = 2 };

template <bool kOn>
struct WaitBeforeExit {
    __device__ ~WaitBeforeExit()
    {
        if constexpr (kOn)
            pdl_wait();
    }
};

template <int RB, int V, Epilogue EP, bool ADD, bool PAIRED, int WAIT = kWaitFirst, bool GF = false>
__global__ void __maxnreg__((reg_cap<RB, V>()))
    fused_rows_kernel(const __grid_constant__ FusedArgs a)
{
    constexpr bool EARLY = WAIT == kEarlyRead;
    const WaitBeforeExit<WAIT == kWaitLast> wait_at_exit;
    static_assert(!PAIRED || V <= 2, "pairs of one- or two-chunk threads");
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const int lane = tid & 31;
    const int64_t row = blockIdx.x;
    const int nc = (int)(a.H >> 3);
    // chunk v of this thread: cbase + v * cstride (tid + v * nthr unpaired;
    // paired, the upper half continues where the lower half's chunks end)
    const int nhalf = nthr >> 1;
    const int cstride = PAIRED ? nhalf : nthr;
    const int cbase = (PAIRED && tid >= nhalf) ? tid + (V - 1) * nhalf : tid;

    // (paired with add_in and 3-4 partials, the 2 x 6 grouped loads would
    // not fit 64 registers beside the pairing: one chunk at a time, still
    // half the sets of loads of the four-chunk layout)
    constexpr int kGroup = (PAIRED && ADD && RB >= 4) ? 1 : load_group<RB, V>();
    constexpr int kE = EARLY ? kGroup : 1;  // early loads held across the wait
    uint4 eraw[kE][EARLY ? RB : 1], eres[kE], eadd[kE];
    if constexpr (EARLY) {
        if (row < a.T) {
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                const int c = cbase + u * cstride;
                if (c < nc) {
                    const int64_t off = row * a.H + (int64_t)c * 8;
#pragma unroll
                    for (int r = 0; r < RB; ++r)
                        if (r < a.R)
                            eraw[u][r] = ld_stream(a.partials[r] + off);
                    if constexpr (EP != Epilogue::kAllReduce) {
                        eres[u] = ld_stream(a.residual + off);
                        if constexpr (ADD)
                            eadd[u] = ld_stream(a.add_in + off);
                    }
                }
            }
        }
    }

    if constexpr (WAIT == kWaitLast)
        pdl_launch_dependents();
    else
        pdl_wait();
    if constexpr (EP == Epilogue::kFp4) {
        if (row >= a.T) {  // a padding row of a swizzled SF buffer: zeros only
            uint8_t *sf = static_cast<uint8_t *>(a.scale_out);
            for (int64_t k4 = tid; k4 < (a.sf_cols >> 2); k4 += nthr)
                st_u32(sf + sf_offset(a, row, k4 * 4), 0u);
            return;
        }
    }

    // With at most 4 partials a CTA keeps too few bytes in flight to cover its
    // own epilogue: it sends the inputs of the row that a CTA one wave later
    // will take (row + prefetch_rows) to L2 with one bulk request per buffer,
    // so DRAM stays busy meanwhile.  Measured gains where the epilogue
    // quantises or R = 1 (NVFP4 R=4 T=16384 H=5120: 153.1 us against 157.4;
    // kARResidualRMSNorm R=1 T=16384 H=7168: 136.7 against 155.7), losses of
    // about 2 % for the bf16 patterns at R = 2..4 and for every R = 8 pattern,
    // which therefore do not prefetch.  For R > 1 the launch enables it only
    // from 3.5 R waves of rows on (launch_rb).
    if constexpr (RB <= 4) {
        constexpr bool kQuant = EP == Epilogue::kFp8Tensor || EP == Epilogue::kFp4 || EP == Epilogue::kFp8Block;
        if ((kQuant || a.R == 1) && tid < 32 && a.prefetch_rows > 0 && row + a.prefetch_rows < a.T) {
            const int64_t pbase = (row + a.prefetch_rows) * a.H;
            const uint32_t bytes = (uint32_t)(a.H * 2);
            if (tid < a.R)
                prefetch_l2(a.partials[tid] + pbase, bytes);
            else if (tid == a.R && EP != Epilogue::kAllReduce)
                prefetch_l2(a.residual + pbase, bytes);
            else if (tid == a.R + 1 && ADD)
                prefetch_l2(a.add_in + pbase, bytes);
        }
    }

    const int64_t rbase = row * a.H;
    float x[V][8];
    float ss = 0.0f;
    // One-chunk threads in calls of at most one wave of rows (paired, or GF)
    // request their gamma chunk with the row's loads, so that it does not
    // wait behind the row reduction: same box, same run, R=8 H=7168 T=16,
    // back to back 2.47 us against 2.62, single cold calls 2.76 against 3.00,
    // and 1.60 against 1.85 with the inputs in L2 and gamma in DRAM (the
    // usual state right after the producing GEMM).  Longer calls keep the
    // load after the reduction: R=2 H=4096 T=16384 measured 97.1 us against
    // 94.4 with it moved.
    constexpr bool kGammaFirst = (PAIRED || GF) && V == 1 && EP != Epilogue::kAllReduce;
    uint4 gfirst = make_uint4(0, 0, 0, 0);
    if constexpr (kGammaFirst) {
        if (cbase < nc)
            gfirst = ld_keep(a.gamma + (int64_t)cbase * 8);
    }

    // ---- phase 1: sum of partials (+ residual), sum of squares ------------
#pragma unroll
    for (int v0 = 0; v0 < V; v0 += kGroup) {
        uint4 raw[kGroup][RB], res[kGroup], addv[kGroup];
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int c = cbase + (v0 + u) * cstride;
            if (EARLY && v0 == 0) {  // loaded before the wait
#pragma unroll
                for (int r = 0; r < RB; ++r)
                    raw[u][r] = eraw[EARLY ? u : 0][EARLY ? r : 0];
                res[u] = eres[EARLY ? u : 0];
                addv[u] = eadd[EARLY ? u : 0];
            } else if (c < nc) {
                const int64_t off = rbase + (int64_t)c * 8;
#pragma unroll
                for (int r = 0; r < RB; ++r)
                    if (r < a.R)
                        raw[u][r] = ld_stream(a.partials[r] + off);
                if constexpr (EP != Epilogue::kAllReduce) {
                    res[u] = ld_stream(a.residual + off);
                    if constexpr (ADD)
                        addv[u] = ld_stream(a.add_in + off);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int v = v0 + u;
            const int c = cbase + v * cstride;
            if (c < nc) {
                const int64_t off = rbase + (int64_t)c * 8;
                float acc[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[e] = 0.0f;
#pragma unroll
                for (int r = 0; r < RB; ++r)
                    if (r < a.R)
                        add_bf16x8(acc, raw[u][r]);
                if (EP == Epilogue::kAllReduce || a.allreduce_out != nullptr)
                    st_v4(a.allreduce_out + off, pack8(acc));
                if constexpr (EP != Epilogue::kAllReduce) {
                    if constexpr (ADD)  // x = ((sum) + add_in) + residual
                        add_bf16x8(acc, addv[u]);
                    add_bf16x8(acc, res[u]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        x[v][e] = acc[e];
                        if constexpr (!PAIRED)
                            ss = fmaf(x[v][e], x[v][e], ss);
                    }
                    st_v4(a.residual_out + off, pack8(x[v]));
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    x[v][e] = 0.0f;
            }
        }
    }
    pdl_launch_dependents();
    if constexpr (EP == Epilogue::kAllReduce)
        return;

    // With two or more chunks per thread, every chunk's gamma is requested
    // before the row reduction: in phase 2 chunk v+1's load would otherwise
    // issue only after chunk v's stores, one dependent L2 round trip per chunk
    // (R=8 T=16 H=7168: 2.59 us per call against 2.85; R=8 T=4096 H=7168:
    // 90.5 us against 91.2).  With one chunk there is no chain to break: a
    // load here, after the row's loads have returned, measured slower (R=2
    // T=16 H=4096: 1.82 us against 1.78), and short calls take the load with
    // the row's loads instead (kGammaFirst above).
    constexpr bool kEarlyGamma = V >= 2 && EP != Epilogue::kAllReduce;
    uint4 gv[V];
    if constexpr (kEarlyGamma) {
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = cbase + v * cstride;
            if (c < nc)
                gv[v] = ld_keep(a.gamma + (int64_t)c * 8);
        }
    }

    if constexpr (PAIRED) {
        __shared__ float carry[kMaxThreadsPaired / 2];
        if (tid < nhalf) {
#pragma unroll
            for (int v = 0; v < V; ++v)
                if (cbase + v * cstride < nc) {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        ss = fmaf(x[v][e], x[v][e], ss);
                }
            carry[tid] = ss;
        }
        __syncthreads();
        if (tid >= nhalf) {
            ss = carry[tid - nhalf];
#pragma unroll
            for (int v = 0; v < V; ++v)
                if (cbase + v * cstride < nc) {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        ss = fmaf(x[v][e], x[v][e], ss);
                }
        }
    }

    // ---- row reduction of x^2 (the same bits in every thread) --------------
    // (paired: the upper half's warps hold the sums, in the lower half's order)
    __shared__ float red[kMaxThreads / 32];
    ss = warp_sum(ss);
    const int nred = PAIRED ? (nthr >> 6) : (nthr >> 5);
    const int wred = PAIRED ? (tid >> 5) - nred : (tid >> 5);
    if (lane == 0 && wred >= 0)
        red[wred] = ss;
    __syncthreads();
    // every warp folds the per-warp sums with the same butterfly, so every
    // thread gets the same bits (each step adds the same two values)
    const float tot = warp_sum(lane < nred ? red[lane] : 0.0f);
    const float scale = rsqrtf(__fadd_rn(__fdiv_rn(tot, (float)a.H), a.eps));

    float qscale = 0.0f;
    if constexpr (EP == Epilogue::kFp8Tensor || EP == Epilogue::kFp4)
        qscale = __ldg(a.scale_factor);
    uint8_t *sf_row = nullptr;  // this row's scale factors (NVFP4)
    int sf_stride = 0;
    if constexpr (EP == Epilogue::kFp4) {
        sf_row = static_cast<uint8_t *>(a.scale_out) + sf_row_base(a, row);
        sf_stride = sf_tile_stride(a);
    }

    // ---- phase 2: norm and the pattern's outputs ----------------------------
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int c = cbase + v * cstride;
        const bool live = c < nc;
        const int64_t off = rbase + (int64_t)c * 8;
        float nf[8];
        uint4 nb = make_uint4(0, 0, 0, 0);
        if (live) {
            float g[8];
            if constexpr (kEarlyGamma)
                unpack8(gv[v], g);
            else if constexpr (kGammaFirst)
                unpack8(gfirst, g);
            else
                unpack8(ld_keep(a.gamma + (int64_t)c * 8), g);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                nf[e] = __fmul_rn(__fmul_rn(x[v][e], scale), g[e]);
            nb = pack8(nf);
            // quantisers read the bf16-rounded n
            unpack8(nb, nf);
            if (a.norm_out != nullptr)
                st_v4(a.norm_out + off, nb);
            if (a.partial_norm_out != nullptr && (int64_t)c * 8 < a.partial_cols)
                st_v4(a.partial_norm_out + row * a.partial_cols + (int64_t)c * 8, nb);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                nf[e] = 0.0f;
        }

        if constexpr (EP == Epilogue::kFp8Tensor) {
            if (live) {
                float q[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    q[e] = __fmul_rn(nf[e], qscale);
                st_v2(a.quant_out + off, cvt_e4m3x8(q));
            }
        } else if constexpr (EP == Epilogue::kFp8Block) {
            float amax = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                amax = fmaxf(amax, fabsf(nf[e]));
            // 16 lanes = 128 columns; all 32 lanes take part in the shuffles
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float sg = div_const_rn(amax, 448.0f, kRcp448);
            if (live) {
                if ((c & 15) == 0)
                    st_f32(static_cast<float *>(a.scale_out) + row * (a.H >> 7) + (c >> 4), sg);
                st_v2(a.quant_out + off, sg != 0.0f ? e4m3_block_codes(nf, sg) : make_uint2(0, 0));
            }
        } else if constexpr (EP == Epilogue::kFp4) {
            float amax = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                amax = fmaxf(amax, fabsf(nf[e]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));  // 16-element block
            const uint32_t sf = cvt_e4m3(__fmul_rn(qscale, div_const_rn(amax, 6.0f, kRcp6)));
            const float d = e4m3_value(sf);
            uint32_t codes = 0;
            if (d != 0.0f) {
                const float es = __fdiv_rn(qscale, d);
                float q[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    q[e] = __fmul_rn(nf[e], es);
                codes = cvt_e2m1x8(q);
            }
            if (live)
                st_u32(a.quant_out + (rbase >> 1) + (int64_t)c * 4, codes);
            // scale factors: SF k = c/2 lives on the even lane; lanes with
            // c % 8 == 0 gather 4 consecutive SFs into one 32-bit store.
            const uint32_t s2 = __shfl_down_sync(0xffffffffu, sf, 2);
            const uint32_t s4 = __shfl_down_sync(0xffffffffu, sf, 4);
            const uint32_t s6 = __shfl_down_sync(0xffffffffu, sf, 6);
            const int k = c >> 1;
            uint8_t *sfk = sf_row + (k >> 2) * sf_stride + (k & 3);
            if (live) {
                if ((a.H & 63) == 0) {
                    if ((lane & 7) == 0)
                        st_u32(sfk, sf | (s2 << 8) | (s4 << 16) | (s6 << 24));
                } else if ((c & 1) == 0) {
                    st_u8(sfk, sf);
                }
            }
        }
    }

    if constexpr (EP == Epilogue::kFp4) {
        // zero the padding columns of this row in the swizzled layout
        if (a.sf_layout != kSfLinear && tid == 0)
            for (int k = (int)(a.H >> 4); k < a.sf_cols; ++k)
                st_u8(sf_row + (k >> 2) * sf_stride + (k & 3), 0u);
    }
}

template <int RB, int V, bool PAIRED = false, int WAIT = kWaitFirst, bool GF = false>
cudaError_t launch_rb_v(Epilogue ep, const FusedArgs &a, int nthr, int64_t grid, bool pdl, cudaStream_t s)
{
    const dim3 g((unsigned)grid), b((unsigned)nthr);
    const bool add = a.add_in != nullptr;  // only with kNorm / kFp8Block (the reduce-scatter Add codes)
    switch (ep) {
    case Epilogue::kAllReduce:
        return launch_kernel(fused_rows_kernel<RB, V, Epilogue::kAllReduce, false, PAIRED, WAIT, GF>, g, b, 0, s, pdl, a);
    case Epilogue::kNorm:
        if (add)
            return launch_kernel(fused_rows_kernel<RB, V, Epilogue::kNorm, true, PAIRED, WAIT, GF>, g, b, 0, s, pdl, a);
        return launch_kernel(fused_rows_kernel<RB, V, Epilogue::kNorm, false, PAIRED, WAIT, GF>, g, b, 0, s, pdl, a);
    case Epilogue::kFp8Tensor:
        return launch_kernel(fused_rows_kernel<RB, V, Epilogue::kFp8Tensor, false, PAIRED, WAIT, GF>, g, b, 0, s, pdl, a);
    case Epilogue::kFp4:
        return launch_kernel(fused_rows_kernel<RB, V, Epilogue::kFp4, false, PAIRED, WAIT, GF>, g, b, 0, s, pdl, a);
    case Epilogue::kFp8Block:
        if (add)
            return launch_kernel(fused_rows_kernel<RB, V, Epilogue::kFp8Block, true, PAIRED, WAIT, GF>, g, b, 0, s, pdl,
                                 a);
        return launch_kernel(fused_rows_kernel<RB, V, Epilogue::kFp8Block, false, PAIRED, WAIT, GF>, g, b, 0, s, pdl, a);
    }
    return cudaErrorInvalidValue;
}

template <int RB>
cudaError_t launch_rb(Epilogue ep, const FusedArgs &a, bool pdl, cudaStream_t s)
{
    const int nc = (int)(a.H >> 3);
    const int V = nc <= kMaxThreads ? 1 : (nc <= 2 * kMaxThreads ? 2 : 4);
    const int per = (nc + V - 1) / V;
    const int nthr = (per + 31) / 32 * 32;
    const int64_t grid = (ep == Epilogue::kFp4 && a.sf_layout != kSfLinear) ? a.sf_rows : a.T;
    const int sms = current_device_sms();
    FusedArgs b = a;
    b.prefetch_rows = 0;
    // Rows that fit one wave of one CTA per SM: each thread of 2 chunks
    // becomes a pair of one-chunk threads, and with at most 4 partials each
    // thread of 4 chunks a pair of two-chunk threads that issue both chunks'
    // loads together, so that a thread waits for fewer sets of loads (same
    // results, see PAIRED).  Single cold calls: R=8 H=7168 T=16 4.08 us
    // against 4.40; NVFP4 R=4 H=12288 T=16 5.28 against 7.07 (3.51 against
    // 4.03 in a CUDA graph).  With 8 partials the four-chunk rows stay
    // unpaired: 4.63 us against 4.18 at H=16384 T=16 in a CUDA graph.
    if constexpr (RB <= 8) {
        if (sms > 0 && a.T <= sms) {
            if (V == 2) return launch_rb_v<RB, 1, true>(ep, b, 2 * nthr, grid, pdl, s);
            if constexpr (RB <= 4) {
                if (V == 4) return launch_rb_v<RB, 2, true>(ep, b, 2 * nthr, grid, pdl, s);
            }
        }
    }
    if (RB <= 4) {  // one wave ahead: SMs x CTAs per SM at the instance's register cap
        if (sms > 0) {
            const int cap = V <= 2 ? reg_cap<RB, 2>() : reg_cap<RB, 4>();
            int per_sm = 65536 / (nthr * cap);
            per_sm = per_sm < 2048 / nthr ? per_sm : 2048 / nthr;
            const int64_t wave = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
            // The first wave's loads queue behind the prefetches of the second
            // wave's R+1 rows, a start-up cost that only enough waves repay.
            // Measured crossovers: R = 1 gains from 9 waves on (H=7168 T=2736:
            // 25.5 us against 28.8); R = 2 is even at 9 waves and gains from 12;
            // R = 4 loses up to 12 waves (NVFP4 H=5120 T=4560: 47.7 against
            // 42.6) and gains from 14.  Hence from 3.5 R waves on, for R > 1.
            if (a.R == 1 || 2 * a.T >= 7 * (int64_t)a.R * wave)
                b.prefetch_rows = wave;
        }
    }
    // TS_FLAG_PDL_EARLY_READ and TS_FLAG_PDL_INDEPENDENT have their own
    // instances for 2 to 8 partials with one or two chunks a thread (the
    // serialised per-rank reduce-scatter calls, FP8 1x128, eight calls of 1024
    // rows at R=8 H=7168: 227.3 us plain, 220.9 early, 188.0 independent; four
    // of 2048 rows at R=4: 139.3, 135.9, 128.7; two of 4096 at R=2: 101.4,
    // 93.8, 98.6 with rank 0 unflagged); elsewhere the flags change nothing
    if constexpr (RB >= 2 && RB <= 8) {
        if (pdl && a.pdl_wait == kEarlyRead) {
            if (V == 1) return launch_rb_v<RB, 1, false, kEarlyRead>(ep, b, nthr, grid, pdl, s);
            if (V == 2) return launch_rb_v<RB, 2, false, kEarlyRead>(ep, b, nthr, grid, pdl, s);
        }
        if (pdl && a.pdl_wait == kWaitLast) {
            if (V == 1) return launch_rb_v<RB, 1, false, kWaitLast>(ep, b, nthr, grid, pdl, s);
            if (V == 2) return launch_rb_v<RB, 2, false, kWaitLast>(ep, b, nthr, grid, pdl, s);
        }
    }
    if (V == 1) {
        if (sms > 0 && grid <= sms)  // gamma with the row's loads (GF)
            return launch_rb_v<RB, 1, false, kWaitFirst, true>(ep, b, nthr, grid, pdl, s);
        return launch_rb_v<RB, 1>(ep, b, nthr, grid, pdl, s);
    }
    if (V == 2) return launch_rb_v<RB, 2>(ep, b, nthr, grid, pdl, s);
    return launch_rb_v<RB, 4>(ep, b, nthr, grid, pdl, s);
}

}  // namespace

cudaError_t launch_fused(Epilogue ep, const FusedArgs &a, bool pdl, cudaStream_t stream)
{
    // the partial loop is unrolled to RB with a predicate per partial, so the
    // small R of tensor parallelism 1 and 2 get their own instances
    if (a.R == 1) return launch_rb<1>(ep, a, pdl, stream);
    if (a.R == 2) return launch_rb<2>(ep, a, pdl, stream);
    if (a.R <= 4) return launch_rb<4>(ep, a, pdl, stream);
    if (a.R <= 8) return launch_rb<8>(ep, a, pdl, stream);
    return launch_rb<16>(ep, a, pdl, stream);
}

}  // namespace tsfn
