// plan.cu -- host-side planning: kernel configuration by shape.  Plain integer
// host code; no CUDA call except the cached SM-count query.
//
// Size classes follow GEMM 优化详解, "矩阵大小选择策略" (small matrices get small
// blocks, large ones large blocks), re-derived for a GPU whose SM count is read at
// run time: the largest tile that still gives every SM a CTA is used.
#include <cuda_runtime.h>

#include <atomic>

#include "fgemm_internal.h"

namespace fgemm {

namespace {

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

}  // namespace

int select_config(int ta, int tb, long long M, long long N, long long K, long long batch,
                  bool aligned, int num_sms)
{
    (void)ta;
    (void)tb;
    if (!aligned) return CFG_64x64_SCALAR;
    if (num_sms < 1) num_sms = 1;
    const long long b = batch > 0 ? batch : 1;
    const long long tiles = ceil_div(M, 128) * ceil_div(N, 128) * b;
    if (tiles >= num_sms) {
        // Two CTAs per SM retire tile-pairs at the rate of lone tiles, so the last
        // r = tiles mod SMs tiles cost a whole lone-tile period.  As quarter tiles
        // they cost ceil(4r / SMs) quarter periods at about 0.7 of the whole-tile
        // rate.  Measured on 152 SMs: a gain for r <= SMs / 2 (FC 8192x4096x11008,
        // r = 32: +1.4 %; 4096x2560x4096, r = 32: +14 %), and for r <= 3/4 SMs when
        // K >= 4096 (4096^3, r = 112: +0.8 %); a loss above 3/4 (3072^3, r = 120:
        // -5.7 %) and at r = 104 with K = 2048 (2048^3: -1.2 %).
        const long long r = tiles % num_sms;
        if (r > 0 && (2 * r <= num_sms || (4 * r <= 3LL * num_sms && K >= 4096)))
            return CFG_128x128_SPLIT;
        return CFG_128x128;
    }
    // 128 x 64 tiles (8 x 8 per thread) beat twice as many 64 x 64 tiles (4 x 4 per
    // thread) as long as they still occupy most SMs (measured: 1024^2, 128 tiles on
    // 152 SMs, 34.8 vs 28.3 TFLOP/s).
    if (ceil_div(M, 128) * ceil_div(N, 64) * b * 5 >= (long long)num_sms * 4) return CFG_128x64;
    // Tiny problems are latency-bound: more, smaller CTAs finish sooner (256^3: 8.2 us
    // with 32 x 32 tiles against 12.4 us with 64 x 64).
    if (ceil_div(M, 64) * ceil_div(N, 64) * b >= num_sms) return CFG_64x64;
    // Up to about two 32 x 32 tiles per SM, four k-groups per tile shorten the serial
    // chain (512^3, 256 tiles: 14.4 us against 16.4 back to back); beyond that the
    // one-group tile wins (768^3, 576 tiles: 35.5 us against 39.6).
    if (ceil_div(M, 32) * ceil_div(N, 32) * b <= 2LL * num_sms) return CFG_32x32_K4;
    return CFG_32x32;
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
