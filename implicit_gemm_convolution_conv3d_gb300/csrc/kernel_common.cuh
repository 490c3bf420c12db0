// kernel_common.cuh -- device helpers shared by the kernel translation units:
// bounded mbarrier waits (every wait in these kernels gives up after a limit
// and records CONV_ERR_TIMEOUT instead of hanging), the bf16 epilogue row
// store, and the per-tensor e4m3 scale and quotient of the fp8 quantisation.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cstdint>

#include "ptx.cuh"

namespace c3d {

constexpr int kStatusTimeout = 4;                     // CONV_ERR_TIMEOUT
constexpr unsigned long long kDrainNs = 1000000000ull;

// The bound is counted in SM clock cycles (clock64 is a cheap SM-local
// register; the global nanosecond timer is far slower to read and would sit on
// every producer / MMA / epilogue hand-off).  Two cycles per nanosecond is the
// SM clock's upper end, so at any lower clock the wall-clock bound only grows.
static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                       int* status, unsigned long long limit_ns) {
    const long long t0 = clock64();
    const long long limit_cycles = static_cast<long long>(limit_ns > (1ull << 61) ? (1ull << 61) : limit_ns) * 2;
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > limit_cycles) {
            *abort_flag = 1u;
            atomicExch(status, kStatusTimeout);
            return false;
        }
    }
}

// Bounded wait on phase `parity` of an mbarrier; false on timeout or abort.
static __device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                         int* status, unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, abort_flag, status, limit_ns);
}

// Cleanup wait: bounded by a fixed limit, ignores the abort flag.
static __device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kDrainNs) return;
    }
}

static __device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Store 32 accumulator columns of one output row (bf16): v * scale + bias
// (bias: the 32 columns' entries, or NULL).
static __device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const uint32_t (&v)[32],
                                               float scale, const float* bias, int count,
                                               bool vec_ok) {
    auto val = [&](int i) {
        return __uint_as_float(v[i]) * scale + (bias ? __ldg(bias + i) : 0.0f);
    };
    if (count == 32 && vec_ok) {
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint4 o;
            o.x = pack_bf16x2(val(8 * i + 0), val(8 * i + 1));
            o.y = pack_bf16x2(val(8 * i + 2), val(8 * i + 3));
            o.z = pack_bf16x2(val(8 * i + 4), val(8 * i + 5));
            o.w = pack_bf16x2(val(8 * i + 6), val(8 * i + 7));
            d4[i] = o;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < count) dst[i] = __float2bfloat16_rn(val(i));
    }
}

// Per-tensor e4m3 scale from the amax word: amax / 448 (IEEE division), 1
// for an all-zero tensor.
static __device__ __forceinline__ float fp8_scale_of(const unsigned int* amax_bits) {
    const float amax = __uint_as_float(*amax_bits);
    return amax == 0.0f ? 1.0f : amax / 448.0f;   // IEEE division (no fast-math)
}

// x / scale correctly rounded, from y = 1/scale correctly rounded (computed
// once): q0 = x*y, r = x - scale*q0 (exact by one FMA), q = q0 + r*y rounded
// once.  This is the FMA correction step of Markstein's division scheme
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Develop. 34(1), 1990): with y the
// correctly rounded reciprocal it returns the correctly rounded quotient
// while no intermediate underflows.  Three instructions where an IEEE
// division takes about three times as many; the pack uses it for scales of
// at least 2^-60 whose significand is not all ones (quotients that matter
// for e4m3 then keep every intermediate far from underflow) and divides
// otherwise.  It runs on |x| and puts x's sign back: for x = -0 the FMAs'
// exact zero sums would give +0 where the division gives -0 (another e4m3
// code).  The exhaustive codec tests compare its codes with the oracle's
// division for every bf16 pattern.
static __device__ __forceinline__ float quot_corrected(float x, float scale, float y) {
    const float xa = fabsf(x);
    const float q0 = __fmul_rn(xa, y);
    const float r = __fmaf_rn(-scale, q0, xa);
    const float q = __fmaf_rn(r, y, q0);
    return __uint_as_float(__float_as_uint(q) | (__float_as_uint(x) & 0x80000000u));
}

// Whether quot_corrected may stand in for the division by this scale.
static __device__ __forceinline__ bool quot_corrected_ok(float scale) {
    return scale >= 8.6736174e-19f &&   // 2^-60
           (__float_as_uint(scale) & 0x7FFFFFu) != 0x7FFFFFu;
}

// Two e4m3 codes (satfinite, round to nearest even) of x0 / scale and
// x1 / scale, x0 in the low byte: the quotient by quot_corrected (CORR) or
// by IEEE division.
template <bool CORR>
static __device__ __forceinline__ uint32_t quant_e4m3x2(float x0, float x1, float scale, float rscale) {
    const float a0 = CORR ? quot_corrected(x0, scale, rscale) : x0 / scale;
    const float a1 = CORR ? quot_corrected(x1, scale, rscale) : x1 / scale;
    return static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(a0, a1), __NV_SATFINITE, __NV_E4M3));
}

}  // namespace c3d
