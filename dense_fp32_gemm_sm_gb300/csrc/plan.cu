// plan.cu -- host-side planning: kernel configuration by shape.  Plain integer
// host code; no CUDA call except the cached SM-count query.
//
// Size classes follow GEMM 优化详解, "矩阵大小选择策略" (small matrices get small
// blocks, large ones large blocks), re-derived for a GPU whose SM count is read at
// run time: each configuration's launch time is estimated from its CTA count per SM
// and K with a fitted model, and the fastest is used.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "fgemm_internal.h"

namespace fgemm {

namespace {

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// Time model of one launch, fitted to CUDA-event times (L2 flushed) of every
// configuration in each transpose layout on 31 shapes (M = N from 256 to 2048 and
// rectangular ones, K from 256 to 4096) on a 152-SM GB300 at 2070 MHz:
//
//     t(us) = a + aK * K + K * max(n * b, L),   n = ceil(CTAs / SMs)
//
// n is the number of CTAs the busiest SM runs (the hardware spreads a grid over
// the SMs breadth-first); b is the time per k of one CTA's share of a busy SM and L
// the per-k latency floor of a CTA that has an SM to itself.  Chosen by the model,
// the fitted shapes lose 0.25 % on average (4.5 % at most) against the fastest
// configuration, and 32 random shapes not used in the fit (all layouts, batches of
// 1 and 3, K from 64 to 6000) 1.4 % on average (27 % at most, one NT shape).  The
// model also predicts 4096^3 (2188 us whole tiles, 2185 us split; measured 2201 and
// 2183), 3072^3, 2048^3 and the FC and PV workloads to within 2 %.
struct LaunchModel {
    double a, aK, b, L;
};
enum ModelSlot { M_128x128, M_128x64, M_64x64, M_32x32, M_32x32_K4, M_QUARTER, NUM_SLOTS };
constexpr LaunchModel kModel[4][NUM_SLOTS] = {
    {  // op(A) N, op(B) N
        {9.26, 0.00815, 0.07485, 0.0000},  // 128x128
        {9.78, -0.00270, 0.04241, 0.0475},  // 128x64
        {7.39, -0.00198, 0.02840, 0.0310},  // 64x64
        {7.30, 0.00285, 0.00781, 0.0140},  // 32x32
        {7.59, -0.00037, 0.00961, 0.0000},  // 32x32 k4
        {10.91, -0.00391, 0.02504, 0.0290},  // quarter
    },
    {  // op(A) N, op(B) T
        {8.77, 0.02036, 0.07595, 0.0000},  // 128x128 (refitted for its 32-deep stages)
        {9.88, 0.00193, 0.04351, 0.0465},  // 128x64
        {6.80, -0.00429, 0.03358, 0.0380},  // 64x64
        {7.15, -0.00007, 0.01026, 0.0185},  // 32x32
        {8.87, -0.00377, 0.01162, 0.0145},  // 32x32 k4
        {10.34, -0.00607, 0.03031, 0.0360},  // quarter
    },
    {  // op(A) T, op(B) N
        {9.35, 0.00555, 0.07214, 0.0000},  // 128x128
        {9.94, -0.02056, 0.04543, 0.0605},  // 128x64
        {7.33, 0.00335, 0.02171, 0.0000},  // 64x64
        {7.57, 0.00052, 0.00588, 0.0170},  // 32x32
        {8.28, -0.00109, 0.00749, 0.0085},  // 32x32 k4
        {10.38, -0.00499, 0.02380, 0.0285},  // quarter
    },
    {  // op(A) T, op(B) T
        {8.99, 0.00259, 0.07926, 0.0000},  // 128x128
        {10.03, 0.00503, 0.03817, 0.0000},  // 128x64
        {7.51, -0.00213, 0.02800, 0.0320},  // 64x64
        {7.52, 0.00109, 0.00790, 0.0150},  // 32x32
        {8.39, -0.00052, 0.00910, 0.0000},  // 32x32 k4
        {10.74, -0.00425, 0.02599, 0.0305},  // quarter
    },
};

double model_n_us(const LaunchModel &m, double n, double K)
{
    const double per_k = n * m.b > m.L ? n * m.b : m.L;
    return m.a + m.aK * K + K * per_k;
}

// CTA counts are products of tile counts and the batch size, which can exceed 64
// bits for arguments the entry points would never see; they are formed in double.
double tiles_of(long long M, long long N, long long bm, long long bn, long long batch)
{
    return (double)ceil_div(M, bm) * (double)ceil_div(N, bn) * (double)batch;
}

double model_us(const LaunchModel &m, double ctas, double K, int num_sms)
{
    return model_n_us(m, std::ceil(ctas / (double)num_sms), K);
}

// Clusters of four k-slice CTAs that run at once with one CTA per SM.  Measured on
// 152 SMs: 74 clusters of four are resident at two CTAs per SM (296 CTAs, not 304:
// a cluster stays inside one GPC), and the k-split tail of r tiles takes
// ceil(r / 37) rounds of a quarter of a whole-tile period.
// The k-chain's cost over the whole-tile model of its S r CTAs at K / S: each of its S
// programmatically dependent launches waits for the one before it to finish before its
// ordered addition into C (8 us a launch), and the model's one launch constant overstates
// a tail whose launches start early (16 us less).  Both fitted to CUDA-event times of
// every slice count 2..8 on 16 shapes on 152 SMs (4096^3, 3072^3, 2048^3, 1024^3, FC,
// PV, TN 3072^2 x 2048, ragged 1700 x 1652, ...): the choice they make is within 0.7 %
// of the fastest slice count and tail on every one.  kTailOverlapUs is the time a
// last-wave launch saves by starting on the SMs the whole tiles leave.
constexpr double kKchainUsPerSlice = 8.0;
constexpr double kKchainCreditUs = 16.0;

// The copy of one operand into the workspace (stage.cu; a transpose or a re-pitch): a
// launch plus its bytes read and written at the copy's measured rate (CUDA events, L2 flushed, on 152 SMs: 64 MB of A at 4096^3
// in 24.6 us, 128 MB in 47.1 us, 16 MB in 9.2 us, 4 MB in 6.1 us).
constexpr double kStageLaunchUs = 4.0;
constexpr double kStageBytesPerUs = 6.2e6;

// Time of the 128 x 128 kernel per k and CTA round in each transpose layout (NN, NT,
// TN, TT), relative to TN, the layout whose two operands both arrive by 16-byte copies.
// Fitted on 152 SMs to whole-tile launches with many CTAs per SM (4096^3 and batched
// 2048 x 2048 problems with K = 128, 256, 512; t = a + n (c + K b)): b = 0.0750 NN,
// 0.0809 NT, 0.0717 TN us; TT measured 4.6 % above TN at K = 128.  The fitted model
// above, from grids of at most a few CTAs per SM, puts the layouts closer together; the
// staging decision compares layouts, so it uses these.
constexpr double kLayoutFactor[4] = {1.046, 1.129, 1.000, 1.046};

// The element-wise configurations against the vector model of their tile.
constexpr double kScalar128 = 1.07;
constexpr double kScalar64 = 1.04;
constexpr double kTailOverlapUs = 35.0;

long long ksplit_clusters_per_round(int num_sms)
{
    const long long c = num_sms / 4 - 1;
    return c > 0 ? c : 1;
}

}  // namespace

int kchain_slices(int ta, int tb, long long r, long long K, int num_sms)
{
    if (num_sms < 1) num_sms = 1;
    const LaunchModel &m = kModel[(ta ? 2 : 0) + (tb ? 1 : 0)][M_128x128];
    const double k = K > 0 ? (double)K : 0.0;
    const double ctas = r > 0 ? (double)r : 0.0;
    int best = 2;
    double best_us = 0.0;
    for (int S = 2; S <= 8; ++S) {
        const double us = model_us(m, S * ctas, k / S, num_sms) + kKchainUsPerSlice * S;
        if (S == 2 || us < best_us) {
            best_us = us;
            best = S;
        }
    }
    return best;
}

double select_config_us(int ta, int tb, long long M, long long N, long long K, long long batch,
                        bool aligned, int num_sms, int *config)
{
    if (num_sms < 1) num_sms = 1;
    if (!aligned) {
        // Element-wise copies: the 128 x 128 tile (whole tiles only) at 1.07x its vector
        // model, or the 64 x 64 tile at 1.04x (measured on 152 SMs, every layout, 256^3 to
        // 4096^3 and the FC, QK^T and PV shapes: the 128 x 128 tile from about 2048^3 up,
        // 1.37x at 4096^3 NN).
        const LaunchModel *const mm = kModel[(ta ? 2 : 0) + (tb ? 1 : 0)];
        const long long b = batch > 0 ? batch : 1;
        const long long k = K > 0 ? K : 0;
        const double s128 = kScalar128 * model_us(mm[M_128x128], tiles_of(M, N, 128, 128, b),
                                                  (double)k, num_sms);
        const double s64 = kScalar64 * model_us(mm[M_64x64], tiles_of(M, N, 64, 64, b),
                                                (double)k, num_sms);
        *config = s128 < s64 ? CFG_128x128_SCALAR : CFG_64x64_SCALAR;
        return s128 < s64 ? s128 : s64;
    }
    const long long b = batch > 0 ? batch : 1;
    const long long k = K > 0 ? K : 0;
    const double tiles128 = tiles_of(M, N, 128, 128, b);
    // The last-wave split: whole 128 x 128 tiles for all but r = tiles mod SMs,
    // then those r as 4r quarter tiles (a second launch; none when r = 0).  r by
    // modular arithmetic, exact for any sizes.
    const long long S = num_sms;
    const long long r = ceil_div(M, 128) % S * (ceil_div(N, 128) % S) % S * (b % S) % S;
    const double whole = tiles128 - (double)r;
    const LaunchModel *const mm = kModel[(ta ? 2 : 0) + (tb ? 1 : 0)];
    const double main_us = whole > 0 ? model_us(mm[M_128x128], whole, k, num_sms) : 0.0;
    // Each last-wave launch is a programmatic dependent of the whole tiles: it starts on
    // the SMs they leave, which hides its launch and the whole tiles' uneven end
    // (measured on 152 SMs: the k-chain 25-40 us below whole tiles + tail model on nine
    // shapes with K from 2048 to 4096).
    // The saving grows with the whole tiles' length (K) up to the measured 35 us.
    const double overlap = whole > 0 ? kTailOverlapUs * (k < 3072 ? (double)k / 3072.0 : 1.0) : 0.0;
    // quarter tiles: 4r CTAs of the quarter model
    const double split = main_us - overlap +
                         (r > 0 ? model_us(mm[M_QUARTER], 4.0 * (double)r, k, num_sms) : 0.0);
    // k-split tiles: whole-tile CTAs over K / 4 each, in rounds of clusters (measured
    // within 2-7 % of the whole-tile model at K / 4 on 152 SMs)
    const double rounds = (double)ceil_div(r, ksplit_clusters_per_round(num_sms));
    const double ksplit = main_us - overlap +
                          (r > 0 ? model_n_us(mm[M_128x128], rounds, (double)k / 4.0) : 0.0);
    // k-chain tiles: S r whole-tile CTAs over K / S each (S from kchain_slices), spread
    // over the SMs without cluster placement, plus the cost of chaining S launches
    const int slices = kchain_slices(ta, tb, r, k, num_sms);
    const double kchain = main_us - overlap +
                          (r > 0 ? model_us(mm[M_128x128], (double)slices * (double)r,
                                            (double)k / slices, num_sms) +
                                       kKchainUsPerSlice * slices - kKchainCreditUs
                                 : 0.0);
    struct Option {
        int config;
        double us;
    };
    const Option options[] = {
        {CFG_128x128, model_us(mm[M_128x128], tiles128, k, num_sms)},
        {CFG_128x128_SPLIT, r > 0 ? split : 1e300},
        {CFG_128x128_KSPLIT, r > 0 ? ksplit : 1e300},
        {CFG_128x128_KCHAIN, r > 0 ? kchain : 1e300},
        {CFG_128x64, model_us(mm[M_128x64], tiles_of(M, N, 128, 64, b), k, num_sms)},
        {CFG_64x64, model_us(mm[M_64x64], tiles_of(M, N, 64, 64, b), k, num_sms)},
        {CFG_32x32, model_us(mm[M_32x32], tiles_of(M, N, 32, 32, b), k, num_sms)},
        {CFG_32x32_K4, model_us(mm[M_32x32_K4], tiles_of(M, N, 32, 32, b), k, num_sms)},
    };
    Option best = options[0];
    for (const Option &o : options)
        if (o.us < best.us) best = o;
    *config = best.config;
    return best.us;
}

int select_config(int ta, int tb, long long M, long long N, long long K, long long batch,
                  bool aligned, int num_sms)
{
    int config = CFG_128x128;
    (void)select_config_us(ta, tb, M, N, K, batch, aligned, num_sms, &config);
    return config;
}

double stage_copy_us(long long R, long long Cc, long long problems)
{
    const double bytes = 8.0 * (double)R * (double)Cc * (double)problems;  // read + write
    return kStageLaunchUs + bytes / kStageBytesPerUs;
}

size_t stage_bytes(int mask, long long M, long long N, long long K, long long problems_a,
                   long long problems_b)
{
    const auto copy = [&](long long rows, long long problems) {
        return sat_mul(sat_mul(sat_mul((size_t)problems, (size_t)K), (size_t)((rows + 3) / 4 * 4)),
                       sizeof(float));
    };
    const size_t a = (mask & 1) ? copy(M, problems_a) : 0;
    const size_t b = (mask & 2) ? copy(N, problems_b) : 0;
    return b == 0 ? a : sat_add(sat_add(a, 255) / 256 * 256, b);
}

int staging_choice(int ta, int tb, long long M, long long N, long long K, long long batch,
                   long long problems_a, long long problems_b, bool aligned_a, bool aligned_b,
                   size_t workspace_bytes, int num_sms)
{
    if (M <= 0 || N <= 0 || K <= 0 || batch <= 0) return 0;
    // A copy can help an operand stored with k contiguous (it is transposed) or one that
    // is k-major but not 16-byte aligned (it gets aligned rows); others stay as stored.
    const int useful = ((ta == 0 || !aligned_a) ? 1 : 0) | ((tb == 1 || !aligned_b) ? 2 : 0);
    if (useful == 0) return 0;
    // Every candidate from one estimate: the GEMM with both operands k-major (op(A) = T,
    // op(B) = N) scaled by the layout's measured cost relative to it; with an unaligned
    // operand left as stored, the element-wise kernels, estimated the same in any layout
    // (their copies move single elements whichever way the operands run: the 128 x 128
    // one measured within 2 % across the four layouts at 4096^3), so a copy that leaves
    // one operand unaligned buys nothing.
    int unused = 0;
    const double base = select_config_us(1, 0, M, N, K, batch, true, num_sms, &unused);
    const double scalar_us = select_config_us(0, 0, M, N, K, batch, false, num_sms, &unused);
    const auto gemm_us = [&](int a, int b, bool aligned) {
        return aligned ? base * kLayoutFactor[(a ? 2 : 0) + (b ? 1 : 0)] : scalar_us;
    };
    // The vector kernels need only the k-major operands aligned (A for op T, B for op N;
    // the others are copied element by element anyway); a copied operand always is.
    const auto vec_ok = [&](int a, int b, bool sa, bool sb) {
        return (sa || a == 0 || aligned_a) && (sb || b == 1 || aligned_b);
    };
    double best_us = gemm_us(ta, tb, vec_ok(ta, tb, false, false));
    int best = 0;
    for (int mask = 1; mask <= 3; ++mask) {
        if ((mask & useful) != mask) continue;
        if (stage_bytes(mask, M, N, K, problems_a, problems_b) > workspace_bytes) continue;
        const bool sa = (mask & 1) != 0, sb = (mask & 2) != 0;
        const int a2 = sa ? 1 : ta, b2 = sb ? 0 : tb;
        double us = gemm_us(a2, b2, vec_ok(a2, b2, sa, sb));
        if (sa) us += stage_copy_us(M, K, problems_a);
        if (sb) us += stage_copy_us(N, K, problems_b);
        // Stage only for a clear gain (1 % and 1 us over the best so far).
        if (us + 0.01 * best_us + 1.0 < best_us) {
            best_us = us;
            best = mask;
        }
    }
    return best;
}

int device_sm_count(int *out)
{
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    const int slot = dev & 63;
    int v = cache[slot].load(std::memory_order_relaxed);
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return -1;
        cache[slot].store(v, std::memory_order_relaxed);
    }
    *out = v;
    return 0;
}

}  // namespace fgemm
