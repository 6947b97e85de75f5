// The C ABI declared in include/ts_fused_norm.h: host-side argument checks,
// then one kernel launch on the caller's stream.  No allocation, no state,
// no synchronisation.
#include <cstdarg>
#include <cstdint>
#include <cstdio>

#include <cuda_runtime.h>

#include "launch.h"
#include "ts_fused_norm.h"

using tsfn::Epilogue;

namespace {

thread_local char g_detail[512];

int fail(int status, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
    va_end(ap);
    return status;
}

int ok()
{
    g_detail[0] = '\0';
    return TS_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// 1/n when n (>= 1) is a power of two, which fp32 holds exactly; else 0.
float pow2_reciprocal(int64_t n)
{
    if (n <= 0 || (n & (n - 1)) != 0)
        return 0.0f;
    float r = 1.0f;
    for (int64_t m = n; m > 1; m >>= 1)
        r *= 0.5f;
    return r;
}

struct Span {
    uintptr_t lo = 0, hi = 0;  // [lo, hi)
    const char *name = "";
};

Span span(const void *p, int64_t bytes, const char *name)
{
    Span s;
    s.lo = reinterpret_cast<uintptr_t>(p);
    s.hi = s.lo + (uintptr_t)(bytes > 0 ? bytes : 0);
    s.name = name;
    return s;
}

bool overlap(const Span &a, const Span &b)
{
    if (a.lo == a.hi || b.lo == b.hi)
        return false;
    return a.lo < b.hi && b.lo < a.hi;
}

// Which outputs each pattern writes: 'R' required, 'o' optional, '-' absent.
// Columns: allreduce_out residual_out norm_out partial_norm_out quant_out scale_out.
const char *const kOutputTable[9] = {
    "R-----",  // 0 kAllReduce
    "oRR---",  // 1 kARResidualRMSNorm
    "oR--R-",  // 2 kARResidualRMSNormFP8Quant
    "oR--RR",  // 3 kARResidualRMSNormFP4Quant
    "oRR-R-",  // 4 kARResidualRMSNormOutFP8Quant
    "oRR-RR",  // 5 kARResidualRMSNormOutFP4Quant
    "oR--RR",  // 6 kARResidualRMSNormFP8BlockWiseQuant
    "oR-RRR",  // 7 kARResidualRMSNormPartialOutFP8BlockWiseQuant
    "oRoR--",  // 8 kARResidualRMSNormPartialOut
};

const char *const kOutputNames[6] = {"allreduce_out", "residual_out", "norm_out",
                                     "partial_norm_out", "quant_out", "scale_out"};

constexpr int64_t kMaxH = 16384;
constexpr uint32_t kKnownFlags = TS_FLAG_PDL;                           // sharded and all-gather norms
constexpr uint32_t kFusedFlags = TS_FLAG_PDL | TS_FLAG_PDL_EARLY_READ | TS_FLAG_PDL_INDEPENDENT;  // fused, RS
constexpr int64_t kMaxRows = 0x7FFFFFFFLL;

}  // namespace

extern "C" const char *ts_status_string(int status)
{
    switch (status) {
    case TS_OK: return "TS_OK";
    case TS_ERR_BAD_PATTERN: return "TS_ERR_BAD_PATTERN";
    case TS_ERR_NULL: return "TS_ERR_NULL";
    case TS_ERR_SHAPE: return "TS_ERR_SHAPE";
    case TS_ERR_ALIGN: return "TS_ERR_ALIGN";
    case TS_ERR_UNSUPPORTED: return "TS_ERR_UNSUPPORTED";
    case TS_ERR_ALIAS: return "TS_ERR_ALIAS";
    case TS_ERR_LAUNCH: return "TS_ERR_LAUNCH";
    default: return "TS_ERR_UNKNOWN";
    }
}

extern "C" const char *ts_last_error_detail(void) { return g_detail; }

namespace {

// Checks and launch of one all-reduce-form pattern (0..8) over T rows.  The
// reduce-scatter entry point lands here too, with the partial pointers
// already moved to the rank's token slice and add_in set for its "Add" codes.
int fused_impl(int pattern, const void *const *partials, int R, const void *add_in, bool needs_add,
               const void *residual, const void *gamma, float eps, const float *scale_factor,
               int64_t T, int64_t H, const ts_outs_t *outs, uint32_t flags, void *stream)
{
    if (outs == nullptr)
        return fail(TS_ERR_NULL, "outs is NULL");
    if (partials == nullptr)
        return fail(TS_ERR_NULL, "partials is NULL");
    if (R < 1 || R > tsfn::kMaxR)
        return fail(TS_ERR_SHAPE, "R = %d outside 1..%d", R, tsfn::kMaxR);
    if (T < 0 || T > kMaxRows)
        return fail(TS_ERR_SHAPE, "T = %lld outside 0..%lld", (long long)T, (long long)kMaxRows);
    if (H < 8 || H % 8 != 0)
        return fail(TS_ERR_SHAPE, "H = %lld must be a positive multiple of 8", (long long)H);
    if (H > kMaxH)
        return fail(TS_ERR_UNSUPPORTED, "H = %lld above the supported maximum %lld", (long long)H,
                    (long long)kMaxH);
    if ((pattern == 6 || pattern == 7) && H % 128 != 0)
        return fail(TS_ERR_SHAPE, "FP8 1x128 blockwise needs H %% 128 == 0 (H = %lld)", (long long)H);
    if ((pattern == 3 || pattern == 5) && H % 16 != 0)
        return fail(TS_ERR_SHAPE, "NVFP4 needs H %% 16 == 0 (H = %lld)", (long long)H);
    if (outs->reserved != 0)
        return fail(TS_ERR_UNSUPPORTED, "ts_outs_t.reserved must be 0");
    if (flags & ~kFusedFlags)
        return fail(TS_ERR_UNSUPPORTED, "unknown flag bits 0x%x", flags & ~kFusedFlags);

    // inputs (with T == 0 the per-row buffers may be NULL: empty tensors)
    const bool empty = T == 0;
    for (int r = 0; r < R; ++r) {
        if (partials[r] == nullptr && !empty)
            return fail(TS_ERR_NULL, "partials[%d] is NULL", r);
        if (!aligned(partials[r], 16))
            return fail(TS_ERR_ALIGN, "partials[%d] is not 16-byte aligned", r);
    }
    if (pattern != 0) {
        if (residual == nullptr && !empty)
            return fail(TS_ERR_NULL, "residual is NULL (required for pattern %d)", pattern);
        if (gamma == nullptr)
            return fail(TS_ERR_NULL, "gamma is NULL (required for pattern %d)", pattern);
        if (!aligned(residual, 16))
            return fail(TS_ERR_ALIGN, "residual is not 16-byte aligned");
        if (!aligned(gamma, 16))
            return fail(TS_ERR_ALIGN, "gamma is not 16-byte aligned");
    }
    if (needs_add) {
        if (add_in == nullptr && !empty)
            return fail(TS_ERR_NULL, "add_in is NULL (required for the reduce-scatter Add patterns)");
        if (!aligned(add_in, 16))
            return fail(TS_ERR_ALIGN, "add_in is not 16-byte aligned");
    } else if (add_in != nullptr) {
        return fail(TS_ERR_UNSUPPORTED, "add_in is only an input of the reduce-scatter Add patterns (7, 8)");
    }
    const bool needs_scale = pattern >= 2 && pattern <= 5;
    if (needs_scale) {
        if (scale_factor == nullptr)
            return fail(TS_ERR_NULL, "scale_factor is NULL (required for pattern %d)", pattern);
        if (!aligned(scale_factor, 4))
            return fail(TS_ERR_ALIGN, "scale_factor is not 4-byte aligned");
    }

    // outputs against the pattern's table
    void *const out_ptr[6] = {outs->allreduce_out, outs->residual_out, outs->norm_out,
                              outs->partial_norm_out, outs->quant_out, outs->scale_out};
    const char *row = kOutputTable[pattern];
    for (int i = 0; i < 6; ++i) {
        if (row[i] == 'R' && out_ptr[i] == nullptr && !empty)
            return fail(TS_ERR_NULL, "%s is required for pattern %d", kOutputNames[i], pattern);
        if (row[i] == '-' && out_ptr[i] != nullptr)
            return fail(TS_ERR_UNSUPPORTED, "%s is not an output of pattern %d (pass NULL)",
                        kOutputNames[i], pattern);
        const uintptr_t need = (i == 5) ? 4 : 16;
        if (out_ptr[i] != nullptr && !aligned(out_ptr[i], need))
            return fail(TS_ERR_ALIGN, "%s is not %d-byte aligned", kOutputNames[i], (int)need);
    }
    const bool fp4 = pattern == 3 || pattern == 5;
    const bool fp8_block = pattern == 6 || pattern == 7;
    const bool partial = pattern == 7 || pattern == 8;
    int64_t P = 0;
    if (partial) {
        P = outs->partial_cols;
        if (P <= 0 || P > H || P % 8 != 0)
            return fail(TS_ERR_SHAPE, "partial_cols = %lld must be in 1..H and a multiple of 8",
                        (long long)P);
    }
    int layout = TS_SF_LINEAR;
    if (fp4) {
        layout = outs->sf_layout;
        if (layout != TS_SF_SWIZZLED_128x4 && layout != TS_SF_SWIZZLED_8x4 && layout != TS_SF_LINEAR)
            return fail(TS_ERR_BAD_PATTERN, "sf_layout %d is not a QuantizationSFLayout code", layout);
    }
    const bool swz = layout != TS_SF_LINEAR;

    // aliasing: outputs disjoint from each other and from the inputs, except
    // allreduce_out == partials[0] and residual_out == residual (in place)
    const int64_t elems = T * H;
    const int64_t n_sf = H / 16;
    const int64_t row_tile = layout == TS_SF_SWIZZLED_128x4 ? 128 : (layout == TS_SF_SWIZZLED_8x4 ? 8 : 1);
    const int64_t sf_rows = (T + row_tile - 1) / row_tile * row_tile;
    const int64_t sf_cols = swz ? (n_sf + 3) / 4 * 4 : n_sf;
    int64_t quant_bytes = fp4 ? elems / 2 : elems;
    int64_t scale_bytes = fp4 ? sf_rows * sf_cols : (fp8_block ? T * (H / 128) * 4 : 0);
    const int64_t out_bytes[6] = {elems * 2, elems * 2, elems * 2, T * P * 2, quant_bytes, scale_bytes};
    Span outs_s[6];
    for (int i = 0; i < 6; ++i)
        outs_s[i] = span(out_ptr[i], out_ptr[i] ? out_bytes[i] : 0, kOutputNames[i]);
    for (int i = 0; i < 6; ++i)
        for (int j = i + 1; j < 6; ++j)
            if (overlap(outs_s[i], outs_s[j]))
                return fail(TS_ERR_ALIAS, "%s overlaps %s", outs_s[i].name, outs_s[j].name);
    for (int i = 0; i < 6; ++i) {
        if (out_ptr[i] == nullptr)
            continue;
        for (int r = 0; r < R; ++r) {
            if (i == 0 && r == 0 && out_ptr[0] == partials[0])
                continue;
            if (overlap(outs_s[i], span(partials[r], elems * 2, "")))
                return fail(TS_ERR_ALIAS, "%s overlaps partials[%d]", kOutputNames[i], r);
        }
        if (pattern != 0) {
            if (!(i == 1 && out_ptr[1] == residual) && overlap(outs_s[i], span(residual, elems * 2, "")))
                return fail(TS_ERR_ALIAS, "%s overlaps residual", kOutputNames[i]);
            if (overlap(outs_s[i], span(gamma, H * 2, "")))
                return fail(TS_ERR_ALIAS, "%s overlaps gamma", kOutputNames[i]);
        }
        if (needs_add && overlap(outs_s[i], span(add_in, elems * 2, "")))
            return fail(TS_ERR_ALIAS, "%s overlaps add_in", kOutputNames[i]);
        if (needs_scale && overlap(outs_s[i], span(scale_factor, 4, "")))
            return fail(TS_ERR_ALIAS, "%s overlaps scale_factor", kOutputNames[i]);
    }

    if (T == 0)
        return ok();

    tsfn::FusedArgs a{};
    for (int r = 0; r < R; ++r)
        a.partials[r] = static_cast<const uint16_t *>(partials[r]);
    a.R = R;
    a.add_in = needs_add ? static_cast<const uint16_t *>(add_in) : nullptr;
    a.residual = static_cast<const uint16_t *>(residual);
    a.gamma = static_cast<const uint16_t *>(gamma);
    a.eps = eps;
    a.scale_factor = needs_scale ? scale_factor : nullptr;
    a.T = T;
    a.H = H;
    a.allreduce_out = static_cast<uint16_t *>(outs->allreduce_out);
    a.residual_out = static_cast<uint16_t *>(outs->residual_out);
    a.norm_out = static_cast<uint16_t *>(outs->norm_out);
    a.partial_norm_out = static_cast<uint16_t *>(outs->partial_norm_out);
    a.partial_cols = P;
    a.quant_out = static_cast<uint8_t *>(outs->quant_out);
    a.scale_out = outs->scale_out;
    a.sf_layout = layout;
    a.sf_rows = sf_rows;
    a.sf_cols = sf_cols;
    const bool pdl = (flags & TS_FLAG_PDL) != 0;
    a.pdl_wait = !pdl ? 0 : (flags & TS_FLAG_PDL_INDEPENDENT) ? 2 : (flags & TS_FLAG_PDL_EARLY_READ) ? 1 : 0;

    Epilogue ep;
    switch (pattern) {
    case 0: ep = Epilogue::kAllReduce; break;
    case 1:
    case 8: ep = Epilogue::kNorm; break;
    case 2:
    case 4: ep = Epilogue::kFp8Tensor; break;
    case 3:
    case 5: ep = Epilogue::kFp4; break;
    default: ep = Epilogue::kFp8Block; break;
    }
    const cudaError_t err = tsfn::launch_fused(ep, a, pdl, static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess)
        return fail(TS_ERR_LAUNCH, "kernel launch failed: %s (%s)", cudaGetErrorName(err),
                    cudaGetErrorString(err));
    return ok();
}

}  // namespace

extern "C" int ts_fused_reduce_norm(int pattern, const void *const *partials, int R,
                                    const void *residual, const void *gamma, float eps,
                                    const float *scale_factor, int64_t T, int64_t H,
                                    const ts_outs_t *outs, uint32_t flags, void *stream)
{
    if (pattern < 0 || pattern > 8)
        return fail(TS_ERR_BAD_PATTERN, "pattern %d is not an AllReduceFusionPattern code (0..8)", pattern);
    return fused_impl(pattern, partials, R, nullptr, false, residual, gamma, eps, scale_factor, T, H, outs,
                      flags, stream);
}

extern "C" int ts_reducescatter_fused_norm(int rs_pattern, const void *const *partials, int R, int rank,
                                           const void *add_in, const void *residual, const void *gamma,
                                           float eps, const float *scale_factor, int64_t T, int64_t H,
                                           const ts_outs_t *outs, uint32_t flags, void *stream)
{
    if (rs_pattern < 0 || rs_pattern > 8)
        return fail(TS_ERR_BAD_PATTERN, "rs_pattern %d is not a ReduceScatterFusionPattern code (0..8)",
                    rs_pattern);
    if (partials == nullptr)
        return fail(TS_ERR_NULL, "partials is NULL");
    if (R < 1 || R > tsfn::kMaxR)
        return fail(TS_ERR_SHAPE, "R = %d outside 1..%d", R, tsfn::kMaxR);
    if (rank < -1 || rank >= R)
        return fail(TS_ERR_SHAPE, "rank = %d outside -1..R-1 (R = %d)", rank, R);
    if (T < 0 || T > kMaxRows)
        return fail(TS_ERR_SHAPE, "T = %lld outside 0..%lld", (long long)T, (long long)kMaxRows);
    if (H < 8 || H % 8 != 0)
        return fail(TS_ERR_SHAPE, "H = %lld must be a positive multiple of 8", (long long)H);
    // token slice of `rank` (T/R each, the first T%R ranks one more); rank -1:
    // every rank's slice, which in rank order is all T tokens
    const int64_t base = T / R, extra = T % R;
    const int64_t count = rank < 0 ? T : base + (rank < extra ? 1 : 0);
    const int64_t start = rank < 0 ? 0 : rank * base + (rank < extra ? rank : extra);
    const void *sliced[tsfn::kMaxR];
    for (int r = 0; r < R; ++r) {
        if (partials[r] == nullptr && T > 0)
            return fail(TS_ERR_NULL, "partials[%d] is NULL", r);
        sliced[r] = partials[r] == nullptr ? nullptr
                                           : static_cast<const uint16_t *>(partials[r]) + start * H;
    }
    const int form = rs_pattern == 7 ? 6 : (rs_pattern == 8 ? 1 : rs_pattern);
    return fused_impl(form, sliced, R, add_in, rs_pattern >= 7, residual, gamma, eps, scale_factor, count, H,
                      outs, flags, stream);
}

namespace {

// Checks and launch shared by ts_qk_norm_sharded and ts_rms_norm_sharded
// (K == 0, no k segment).
int sharded_norm(const char *what, const void *const *shards, int R, int64_t T, int64_t row_stride,
                 int64_t Q, int64_t K, const void *q_weight, const void *k_weight, float eps,
                 void *q_out, int64_t ldq, void *k_out, int64_t ldk, uint32_t flags, void *stream)
{
    const bool has_k = K != 0;
    if (shards == nullptr)
        return fail(TS_ERR_NULL, "%s is NULL", what);
    if (R < 1 || R > tsfn::kMaxR)
        return fail(TS_ERR_SHAPE, "R = %d outside 1..%d", R, tsfn::kMaxR);
    if (T < 0 || T > kMaxRows)
        return fail(TS_ERR_SHAPE, "T = %lld outside 0..%lld", (long long)T, (long long)kMaxRows);
    if (flags & ~kKnownFlags)
        return fail(TS_ERR_UNSUPPORTED, "unknown flag bits 0x%x", flags & ~kKnownFlags);
    if (Q < 8 || Q % 8 != 0 || (has_k && (K < 8 || K % 8 != 0)))
        return fail(TS_ERR_SHAPE, "segment widths (%lld, %lld) must be positive multiples of 8",
                    (long long)Q, (long long)K);
    if (Q > 4096 || K > 1024)
        return fail(TS_ERR_UNSUPPORTED, "segment widths up to 4096 (q / single) and 1024 (k) are supported");
    if (row_stride % 8 != 0 || row_stride < Q + K)
        return fail(TS_ERR_SHAPE, "row_stride = %lld must be a multiple of 8 and cover the segments",
                    (long long)row_stride);
    if (ldq % 8 != 0 || ldq < R * Q)
        return fail(TS_ERR_SHAPE, "output leading dimension %lld must be a multiple of 8 and >= R*width",
                    (long long)ldq);
    if (has_k && (ldk % 8 != 0 || ldk < R * K))
        return fail(TS_ERR_SHAPE, "ldk = %lld must be a multiple of 8 and >= R*k_shard", (long long)ldk);
    const bool empty = T == 0;  // per-token buffers may then be NULL (empty tensors)
    for (int r = 0; r < R; ++r) {
        if (shards[r] == nullptr && !empty)
            return fail(TS_ERR_NULL, "%s[%d] is NULL", what, r);
        if (!aligned(shards[r], 16))
            return fail(TS_ERR_ALIGN, "%s[%d] is not 16-byte aligned", what, r);
    }
    const void *const ptrs[4] = {q_weight, k_weight, q_out, k_out};
    const char *const names[4] = {has_k ? "q_weight" : "weight", "k_weight", has_k ? "q_out" : "out", "k_out"};
    for (int i = 0; i < 4; ++i) {
        if (!has_k && (i == 1 || i == 3))
            continue;
        if (ptrs[i] == nullptr && !(empty && i >= 2))
            return fail(TS_ERR_NULL, "%s is NULL", names[i]);
        if (!aligned(ptrs[i], 16))
            return fail(TS_ERR_ALIGN, "%s is not 16-byte aligned", names[i]);
    }
    if (T > 0) {
        const Span qo = span(q_out, ((T - 1) * ldq + R * Q) * 2, names[2]);
        const Span ko = span(has_k ? k_out : nullptr, has_k ? ((T - 1) * ldk + R * K) * 2 : 0, "k_out");
        if (overlap(qo, ko))
            return fail(TS_ERR_ALIAS, "q_out overlaps k_out");
        const Span ins[2] = {span(q_weight, R * Q * 2, names[0]),
                             span(has_k ? k_weight : nullptr, R * K * 2, "k_weight")};
        for (const Span &o : {qo, ko}) {
            for (const Span &in : ins)
                if (overlap(o, in))
                    return fail(TS_ERR_ALIAS, "%s overlaps %s", o.name, in.name);
            for (int r = 0; r < R; ++r)
                if (overlap(o, span(shards[r], ((T - 1) * row_stride + Q + K) * 2, "")))
                    return fail(TS_ERR_ALIAS, "%s overlaps %s[%d]", o.name, what, r);
        }
    }
    if (T == 0)
        return ok();

    tsfn::QKArgs a{};
    for (int r = 0; r < R; ++r)
        a.shards[r] = static_cast<const uint16_t *>(shards[r]);
    a.R = R;
    a.div_r = tsfn::div_magic((uint32_t)R);
    a.T = T;
    a.row_stride = row_stride;
    a.Q = (int)Q;
    a.K = (int)K;
    a.inv_q = pow2_reciprocal(Q);
    a.inv_k = pow2_reciprocal(K);
    a.inv_r = pow2_reciprocal(R);
    a.q_weight = static_cast<const uint16_t *>(q_weight);
    a.k_weight = has_k ? static_cast<const uint16_t *>(k_weight) : nullptr;
    a.eps = eps;
    a.q_out = static_cast<uint16_t *>(q_out);
    a.ldq = ldq;
    a.k_out = has_k ? static_cast<uint16_t *>(k_out) : nullptr;
    a.ldk = has_k ? ldk : 0;
    const cudaError_t err =
        tsfn::launch_qk(a, (flags & TS_FLAG_PDL) != 0, static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess)
        return fail(TS_ERR_LAUNCH, "kernel launch failed: %s (%s)", cudaGetErrorName(err),
                    cudaGetErrorString(err));
    return ok();
}

}  // namespace

extern "C" int ts_qk_norm_sharded(const void *const *qkv_shards, int R, int64_t T,
                                  int64_t row_stride, int64_t q_shard, int64_t k_shard,
                                  const void *q_weight, const void *k_weight, float eps,
                                  void *q_out, int64_t ldq, void *k_out, int64_t ldk, uint32_t flags,
                                  void *stream)
{
    if (k_shard == 0)
        return fail(TS_ERR_SHAPE, "k_shard must be a positive multiple of 8 (use ts_rms_norm_sharded for one segment)");
    return sharded_norm("qkv_shards", qkv_shards, R, T, row_stride, q_shard, k_shard, q_weight, k_weight,
                        eps, q_out, ldq, k_out, ldk, flags, stream);
}

extern "C" int ts_rms_norm_sharded(const void *const *shards, int R, int64_t T, int64_t row_stride,
                                   int64_t width, const void *weight, float eps, void *out, int64_t ldo,
                                   uint32_t flags, void *stream)
{
    return sharded_norm("shards", shards, R, T, row_stride, width, 0, weight, nullptr, eps, out, ldo,
                        nullptr, 0, flags, stream);
}

extern "C" int ts_allgather_fused_norm(int ag_pattern, const void *const *inputs, int R, int64_t T,
                                       int64_t hidden, int64_t q_lora_rank, int64_t kv_lora_rank,
                                       int64_t qk_rope_head_dim, const void *x_gamma, const void *y_gamma,
                                       float x_eps, float y_eps, void *allgather_out, void *x_norm_out,
                                       void *y_norm_out, void *quant_out, void *scale_out, uint32_t flags,
                                       void *stream)
{
    if (ag_pattern < 0 || ag_pattern > 2)
        return fail(TS_ERR_BAD_PATTERN, "ag_pattern %d is not an AllGatherFusionPattern code (0..2)", ag_pattern);
    if (inputs == nullptr)
        return fail(TS_ERR_NULL, "inputs is NULL");
    if (R < 1 || R > tsfn::kMaxR)
        return fail(TS_ERR_SHAPE, "R = %d outside 1..%d", R, tsfn::kMaxR);
    if (T < 0 || T > kMaxRows)
        return fail(TS_ERR_SHAPE, "T = %lld outside 0..%lld", (long long)T, (long long)kMaxRows);
    if (flags & ~kKnownFlags)
        return fail(TS_ERR_UNSUPPORTED, "unknown flag bits 0x%x", flags & ~kKnownFlags);
    const int64_t q = q_lora_rank, kv = kv_lora_rank, rope = qk_rope_head_dim;
    if (q <= 0 || q % 128 != 0)
        return fail(TS_ERR_SHAPE, "q_lora_rank = %lld must be a positive multiple of 128", (long long)q);
    if (kv <= 0 || kv % 8 != 0 || rope < 0 || rope % 8 != 0)
        return fail(TS_ERR_SHAPE, "kv_lora_rank (%lld) and qk_rope_head_dim (%lld) must be multiples of 8",
                    (long long)kv, (long long)rope);
    if (q + kv + rope != hidden)
        return fail(TS_ERR_SHAPE, "q_lora_rank + kv_lora_rank + qk_rope_head_dim (%lld) != hidden (%lld)",
                    (long long)(q + kv + rope), (long long)hidden);
    if (hidden > 2112)
        return fail(TS_ERR_SHAPE, "hidden = %lld above 2112", (long long)hidden);
    const bool empty = T == 0;
    const int64_t base = T / R, extra = T % R;
    for (int r = 0; r < R; ++r) {
        const int64_t count = base + (r < extra ? 1 : 0);
        if (inputs[r] == nullptr && count > 0)
            return fail(TS_ERR_NULL, "inputs[%d] is NULL", r);
        if (!aligned(inputs[r], 16))
            return fail(TS_ERR_ALIGN, "inputs[%d] is not 16-byte aligned", r);
    }
    if (ag_pattern != 0) {
        if (x_gamma == nullptr || y_gamma == nullptr)
            return fail(TS_ERR_NULL, "x_gamma and y_gamma are required for pattern %d", ag_pattern);
        if (!aligned(x_gamma, 16) || !aligned(y_gamma, 16))
            return fail(TS_ERR_ALIGN, "x_gamma / y_gamma are not 16-byte aligned");
    }
    // outputs: allgather_out always; x_norm_out 1 (optional in 2); y_norm_out 1, 2; quant/scale 2
    void *const outp[5] = {allgather_out, x_norm_out, y_norm_out, quant_out, scale_out};
    const char *const names[5] = {"allgather_out", "x_norm_out", "y_norm_out", "quant_out", "scale_out"};
    const char *const table[3] = {"R----", "RRR--", "RoRRR"};
    for (int i = 0; i < 5; ++i) {
        const char need = table[ag_pattern][i];
        if (need == 'R' && outp[i] == nullptr && !empty)
            return fail(TS_ERR_NULL, "%s is required for pattern %d", names[i], ag_pattern);
        if (need == '-' && outp[i] != nullptr)
            return fail(TS_ERR_UNSUPPORTED, "%s is not an output of pattern %d (pass NULL)", names[i], ag_pattern);
        if (outp[i] != nullptr && !aligned(outp[i], i == 4 ? 4 : 16))
            return fail(TS_ERR_ALIGN, "%s is not %d-byte aligned", names[i], i == 4 ? 4 : 16);
    }
    if (empty)
        return ok();
    const int64_t out_bytes[5] = {T * hidden * 2, T * q * 2, T * kv * 2, T * q, T * (q / 128) * 4};
    Span os[5];
    for (int i = 0; i < 5; ++i)
        os[i] = span(outp[i], outp[i] ? out_bytes[i] : 0, names[i]);
    for (int i = 0; i < 5; ++i) {
        for (int j = i + 1; j < 5; ++j)
            if (overlap(os[i], os[j]))
                return fail(TS_ERR_ALIAS, "%s overlaps %s", os[i].name, os[j].name);
        for (int r = 0; r < R; ++r)
            if (overlap(os[i], span(inputs[r], (base + (r < extra ? 1 : 0)) * hidden * 2, "")))
                return fail(TS_ERR_ALIAS, "%s overlaps inputs[%d]", os[i].name, r);
        if (ag_pattern != 0 && (overlap(os[i], span(x_gamma, q * 2, "")) || overlap(os[i], span(y_gamma, kv * 2, ""))))
            return fail(TS_ERR_ALIAS, "%s overlaps a gamma", os[i].name);
    }

    tsfn::AGArgs a{};
    for (int r = 0; r < R; ++r)
        a.inputs[r] = static_cast<const uint16_t *>(inputs[r]);
    a.R = R;
    a.T = T;
    a.base = (uint32_t)base;
    a.extra = (uint32_t)extra;
    a.split = (uint32_t)(extra * (base + 1));
    a.div_hi = tsfn::div_magic((uint32_t)(base + 1));
    a.div_lo = tsfn::div_magic(base > 0 ? (uint32_t)base : 1u);
    a.hidden = (int)hidden;
    a.q = (int)q;
    a.kv = (int)kv;
    a.x_gamma = static_cast<const uint16_t *>(x_gamma);
    a.y_gamma = static_cast<const uint16_t *>(y_gamma);
    a.x_eps = x_eps;
    a.y_eps = y_eps;
    a.pattern = ag_pattern;
    a.allgather_out = static_cast<uint16_t *>(allgather_out);
    a.x_norm_out = static_cast<uint16_t *>(x_norm_out);
    a.y_norm_out = static_cast<uint16_t *>(y_norm_out);
    a.quant_out = static_cast<uint8_t *>(quant_out);
    a.scale_out = static_cast<float *>(scale_out);
    const cudaError_t err = tsfn::launch_ag(a, (flags & TS_FLAG_PDL) != 0, static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess)
        return fail(TS_ERR_LAUNCH, "kernel launch failed: %s (%s)", cudaGetErrorName(err), cudaGetErrorString(err));
    return ok();
}
