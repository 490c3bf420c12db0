// aux_kernels.cu -- HBM-bound kernels around the convolution:
//   * split-K reduction (FlyDSL PR #860, split-K commits): fp32 partials
//     summed in fixed split order, scaled, rounded to bf16;
//   * amax of a bf16 tensor, and the tiled NCDHW -> NDHWC pack with optional
//     per-tensor fp8-e4m3 quantisation (FlyDSL PR #860, commit adding the
//     tiled bf16 -> fp8 transpose that replaces torch.permute, and the commit
//     fixing its >2 GB addressing with 64-bit offsets).
#include <cuda_bf16.h>
#include <cuda_fp8.h>


#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace c3d {

namespace {

// ----------------------------------------------------------------- split-K
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ ws,
                                                            __nv_bfloat16* __restrict__ out,
                                                            long long MK, int splits,
                                                            const float* scale_x,
                                                            const float* scale_w,
                                                            const float* bias, long long K,
                                                            int act) {
    float scale = 1.0f;
    if (scale_x) scale *= *scale_x;
    if (scale_w) scale *= *scale_w;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if ((MK & 3) == 0) {
        const long long n4 = MK >> 2;
        for (long long i = tid; i < n4; i += stride) {
            float4 acc = reinterpret_cast<const float4*>(ws)[i];
            for (int s = 1; s < splits; ++s) {
                const float4 v = reinterpret_cast<const float4*>(ws + s * MK)[i];
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            float b[4] = {0.f, 0.f, 0.f, 0.f};
            if (bias) {
                const long long k0 = (i << 2) % K;
#pragma unroll
                for (int j = 0; j < 4; ++j) b[j] = __ldg(bias + (k0 + j) % K);
            }
            __nv_bfloat162 lo = __floats2bfloat162_rn(activate(acc.x * scale + b[0], act),
                                                      activate(acc.y * scale + b[1], act));
            __nv_bfloat162 hi = __floats2bfloat162_rn(activate(acc.z * scale + b[2], act),
                                                      activate(acc.w * scale + b[3], act));
            uint2 o;
            o.x = *reinterpret_cast<uint32_t*>(&lo);
            o.y = *reinterpret_cast<uint32_t*>(&hi);
            reinterpret_cast<uint2*>(out)[i] = o;
        }
    } else {
        for (long long i = tid; i < MK; i += stride) {
            float acc = ws[i];
            for (int s = 1; s < splits; ++s) acc += ws[s * MK + i];
            out[i] = __float2bfloat16_rn(
                activate(acc * scale + (bias ? __ldg(bias + i % K) : 0.f), act));
        }
    }
}

// ----------------------------------------------------------------- amax
// max |x| of a bf16 tensor into *amax_bits (the bit pattern of a non-negative
// binary32 orders like an unsigned integer, so atomicMax on the bits is the
// float max).  *amax_bits must be zero before the launch.
__global__ void __launch_bounds__(256) amax_bf16_kernel(const __nv_bfloat16* __restrict__ in,
                                                        long long n, unsigned int* amax_bits) {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    unsigned int m = 0;   // max over |x| as bf16 magnitude bits
    const long long n8 = n >> 3;
    const uint4* in8 = reinterpret_cast<const uint4*>(in);
    for (long long i = tid; i < n8; i += stride) {
        const uint4 v = __ldcs(in8 + i);
        const unsigned int w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            m = max(m, w[j] & 0x7FFFu);
            m = max(m, (w[j] >> 16) & 0x7FFFu);
        }
    }
    const unsigned short* in16 = reinterpret_cast<const unsigned short*>(in);
    for (long long i = (n8 << 3) + tid; i < n; i += stride) m = max(m, in16[i] & 0x7FFFu);
    // bf16 magnitude bits << 16 are the binary32 bits of the same value
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    __shared__ unsigned int red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned int b = 0;
        for (int i = 0; i < (blockDim.x >> 5); ++i) b = max(b, red[i]);
        atomicMax(amax_bits, b << 16);
    }
}

// ----------------------------------------------------------------- pack
// One CTA moves a tile of 64 channels x 64 spatial positions of one image:
// coalesced reads of 64 rows of 64 spatial values (128 B each) into shared
// memory, then each thread emits 16 consecutive channels of one spatial
// position (16 B of fp8 or 32 B of bf16), four threads covering a 64-channel
// run.  All offsets are 64-bit.
constexpr int kPackC = 64;
constexpr int kPackS = 64;
constexpr int kPitch = kPackS + 2;   // bf16 elements per smem row (33 words: no bank conflicts)


template <int FP8>
__global__ void __launch_bounds__(256) pack_kernel(const __nv_bfloat16* __restrict__ in,
                                                   long long N, long long C, long long S,
                                                   void* __restrict__ out,
                                                   const unsigned int* amax_bits,
                                                   float* scale_out, long long c_tiles,
                                                   long long s_tiles) {
    griddep_launch_dependents();   // the conv reading this output waits for completion
    __shared__ __align__(16) unsigned short tile[kPackC * kPitch];
    const long long b = blockIdx.x;
    const long long st = b % s_tiles;
    const long long rest = b / s_tiles;
    const long long ct = rest % c_tiles;
    const long long n = rest / c_tiles;
    const long long s0 = st * kPackS, c0 = ct * kPackC;
    const unsigned short* src = reinterpret_cast<const unsigned short*>(in);

    // load: 64 channel rows x 64 positions; thread -> (row, 8-position piece)
    const bool vec_in = (S % 8) == 0;
    for (int i = threadIdx.x; i < kPackC * (kPackS / 8); i += blockDim.x) {
        const int r = i >> 3, piece = i & 7;
        const long long c = c0 + r, s = s0 + piece * 8;
        unsigned short v[8];
        if (c < C && vec_in && s + 8 <= S) {
            const uint4 q = __ldcs(reinterpret_cast<const uint4*>(src + (n * C + c) * S + s));
            const unsigned int w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[2 * j] = static_cast<unsigned short>(w[j] & 0xFFFFu);
                v[2 * j + 1] = static_cast<unsigned short>(w[j] >> 16);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = (c < C && s + j < S) ? src[(n * C + c) * S + s + j] : 0;
        }
        unsigned int* trow = reinterpret_cast<unsigned int*>(tile + r * kPitch + piece * 8);
#pragma unroll
        for (int j = 0; j < 4; ++j) trow[j] = static_cast<unsigned int>(v[2 * j]) |
                                              (static_cast<unsigned int>(v[2 * j + 1]) << 16);
    }
    __syncthreads();

    float scale = 1.0f;
    if (FP8) {
        scale = fp8_scale_of(amax_bits);
        if (b == 0 && threadIdx.x == 0) *scale_out = scale;
    }
    // store: thread -> (position, 16-channel group)
    const int g = threadIdx.x & 3;
    for (int sp = threadIdx.x >> 2; sp < kPackS; sp += blockDim.x >> 2) {
        const long long s = s0 + sp;
        const long long cb = c0 + g * 16;
        if (s >= S || cb >= C) continue;
        unsigned short v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = tile[(g * 16 + j) * kPitch + sp];
        const long long obase = (n * S + s) * C + cb;
        const bool full = (cb + 16 <= C);
        if (FP8) {
            unsigned char* o = reinterpret_cast<unsigned char*>(out);
            unsigned char q[16];
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                const float a = __uint_as_float(static_cast<unsigned int>(v[j]) << 16) / scale;
                const float c2 = __uint_as_float(static_cast<unsigned int>(v[j + 1]) << 16) / scale;
                const __nv_fp8x2_storage_t p2 =
                    __nv_cvt_float2_to_fp8x2(make_float2(a, c2), __NV_SATFINITE, __NV_E4M3);
                q[j] = static_cast<unsigned char>(p2 & 0xFFu);
                q[j + 1] = static_cast<unsigned char>(p2 >> 8);
            }
            if (full && (C % 16) == 0) {
                uint4 w;
                w.x = q[0] | (q[1] << 8) | (q[2] << 16) | (static_cast<unsigned int>(q[3]) << 24);
                w.y = q[4] | (q[5] << 8) | (q[6] << 16) | (static_cast<unsigned int>(q[7]) << 24);
                w.z = q[8] | (q[9] << 8) | (q[10] << 16) | (static_cast<unsigned int>(q[11]) << 24);
                w.w = q[12] | (q[13] << 8) | (q[14] << 16) | (static_cast<unsigned int>(q[15]) << 24);
                *reinterpret_cast<uint4*>(o + obase) = w;
            } else {
                for (int j = 0; j < 16 && cb + j < C; ++j) o[obase + j] = q[j];
            }
        } else {
            unsigned short* o = reinterpret_cast<unsigned short*>(out);
            if (full && (C % 8) == 0) {
                uint4 w0, w1;
                w0.x = v[0] | (v[1] << 16);
                w0.y = v[2] | (v[3] << 16);
                w0.z = v[4] | (v[5] << 16);
                w0.w = v[6] | (v[7] << 16);
                w1.x = v[8] | (v[9] << 16);
                w1.y = v[10] | (v[11] << 16);
                w1.z = v[12] | (v[13] << 16);
                w1.w = v[14] | (v[15] << 16);
                reinterpret_cast<uint4*>(o + obase)[0] = w0;
                reinterpret_cast<uint4*>(o + obase)[1] = w1;
            } else {
                for (int j = 0; j < 16 && cb + j < C; ++j) o[obase + j] = v[j];
            }
        }
    }
}

// Register-blocked pack for the regular case (C % 16 == 0, S % 8 == 0):
// each thread owns 16 channels x 8 consecutive positions.  It reads the 16
// channel rows with one 16-byte load each, transposes in registers, and
// writes each position's 16 channels as one 16-byte (fp8) or two 16-byte
// (bf16) stores; LC lanes cover a 16*LC-channel run of one position.  A warp
// covers 16*LC channels x 256/LC positions; the grid is persistent and walks
// tiles.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int FP8, int LC>
__global__ void __launch_bounds__(256) pack_tiles_kernel(const __nv_bfloat16* __restrict__ in,
                                                         long long C, long long S,
                                                         void* __restrict__ out,
                                                         const unsigned int* amax_bits,
                                                         float* scale_out, long long c_tiles,
                                                         long long s_tiles, long long tiles) {
    griddep_launch_dependents();   // the conv reading this output waits for completion
    float scale = 1.0f;
    if (FP8) {
        scale = fp8_scale_of(amax_bits);
        if (blockIdx.x == 0 && threadIdx.x == 0) *scale_out = scale;
    }
    const int lane = threadIdx.x & 31;
    // LC lanes cover one position's 16*LC channels; a warp covers 16*LC
    // channels x 256/LC positions
    const int cg = lane % LC, sb = lane / LC;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    for (long long tile = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         tile < tiles; tile += warps) {
        // channel tiles fastest: the warps that write the other channels of
        // the same output positions run at the same time, so each output
        // line is completed in L2 before it is written back
        const long long ct = tile % c_tiles;
        const long long rest = tile / c_tiles;
        const long long st = rest % s_tiles;
        const long long n = rest / s_tiles;
        const long long c0 = ct * (16 * LC) + cg * 16;
        const long long s0 = st * (256 / LC) + sb * 8;
        if (c0 >= C || s0 >= S) continue;
        uint4 v[16];
        const __nv_bfloat16* src = in + (n * C + c0) * S + s0;
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __ldcs(reinterpret_cast<const uint4*>(src + j * S));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            // element i of each row: word i/2, low or high half
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const uint32_t ww = (i >> 1) == 0 ? v[j].x : (i >> 1) == 1 ? v[j].y : (i >> 1) == 2 ? v[j].z : v[j].w;
                w[j] = ww;
            }
            const long long obase = (n * S + s0 + i) * C + c0;
            if (FP8) {
                uint32_t o[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uint32_t b = 0;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int j = 4 * k + 2 * h;
                        const float a0 = ((i & 1) ? bf16_hi(w[j]) : bf16_lo(w[j])) / scale;
                        const float a1 = ((i & 1) ? bf16_hi(w[j + 1]) : bf16_lo(w[j + 1])) / scale;
                        const __nv_fp8x2_storage_t q2 =
                            __nv_cvt_float2_to_fp8x2(make_float2(a0, a1), __NV_SATFINITE, __NV_E4M3);
                        b |= static_cast<uint32_t>(q2) << (16 * h);
                    }
                    o[k] = b;
                }
                *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(out) + obase) =
                    make_uint4(o[0], o[1], o[2], o[3]);
            } else {
                uint32_t o[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t e0 = (i & 1) ? (w[2 * k] >> 16) : (w[2 * k] & 0xFFFFu);
                    const uint32_t e1 = (i & 1) ? (w[2 * k + 1] >> 16) : (w[2 * k + 1] & 0xFFFFu);
                    o[k] = e0 | (e1 << 16);
                }
                uint4* d = reinterpret_cast<uint4*>(reinterpret_cast<unsigned short*>(out) + obase);
                d[0] = make_uint4(o[0], o[1], o[2], o[3]);
                d[1] = make_uint4(o[4], o[5], o[6], o[7]);
            }
        }
    }
}

// ----------------------------------------------------------------- TMA-fed pack
// The pack for C % 8 == 0 and D*H*W % 8 == 0 with the activation arriving by
// TMA.  Per image the input is a [C, S] matrix (S = D*H*W positions); a tile
// is 128 channel rows x 256 positions: 512 contiguous bytes of each row, one
// TMA box {256, 128, 1} (out-of-range rows and positions read as zeros and
// are not stored).  One producer thread keeps `stages` tiles in flight in a
// shared-memory ring (full / empty mbarriers), so the bytes in flight sit in
// shared memory, not in registers.  Sixteen converter warps transpose each
// tile in units of 8 channels x 8 positions, one unit per thread: eight
// 16-byte row reads -- conflict-free, the 8 lanes of a quarter-warp read 8
// consecutive 16-byte pieces of one row -- then each position's 8 channels
// leave as one 8-byte (e4m3) or 16-byte (bf16) store.  Persistent grid;
// tiles are walked channels-fastest, so the CTAs running together write all
// channels of the same output positions (whole output rows leave L2
// together) while each reads 512-byte pieces of its channel rows.
constexpr int kTmaPackPos = 256;
constexpr int kTmaPackConvWarps = 16;
constexpr int kTmaPackThreads = (kTmaPackConvWarps + 1) * 32;
constexpr unsigned long long kPackDrainCycles = 2000000000ull;

template <int FP8>
struct TmaPackShape {
    static constexpr int kC = 128;                                  // channels per tile
    static constexpr uint32_t kStageBytes = kC * kTmaPackPos * 2;   // bf16 input tile
};

// Bounded mbarrier wait of the pack kernel: false once the abort flag is set
// or the limit (SM cycles at 2 per ns) passes, recording the timeout.
__device__ __noinline__ bool pack_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                       int* status, unsigned long long limit_ns) {
    const long long t0 = clock64();
    const long long limit = static_cast<long long>(limit_ns > (1ull << 61) ? (1ull << 61) : limit_ns) * 2;
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) {
            *abort_flag = 1u;
            atomicExch(status, 4);   // CONV_ERR_TIMEOUT
            return false;
        }
    }
    return true;
}

// One converter unit of the TMA-fed pack: 8 channel rows x 8 positions of the
// tile in shared memory (v: row k's 8 positions) to 8 output positions.
template <int FP8, bool CORR>
__device__ __forceinline__ void pack_unit_store(const uint4 (&v)[8], long long n, long long s0,
                                                long long c, long long C, long long S, void* out,
                                                float scale, float rscale) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const long long s = s0 + i;
        if (s >= S) break;
        // element i of each channel row: word i/2, low or high half
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t ww = (i >> 1) == 0 ? v[k].x : (i >> 1) == 1 ? v[k].y
                              : (i >> 1) == 2 ? v[k].z : v[k].w;
            w[k] = (i & 1) ? (ww >> 16) : (ww & 0xFFFFu);
        }
        const long long o = (n * S + s) * C + c;
        if (FP8) {
            uint32_t q[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t b = 0;
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    b |= quant_e4m3x2<CORR>(__uint_as_float(w[4 * h + e] << 16),
                                            __uint_as_float(w[4 * h + e + 1] << 16), scale,
                                            rscale) << (8 * e);
                }
                q[h] = b;
            }
            *reinterpret_cast<uint2*>(static_cast<unsigned char*>(out) + o) = make_uint2(q[0], q[1]);
        } else {
            *reinterpret_cast<uint4*>(static_cast<unsigned short*>(out) + o) =
                make_uint4(w[0] | (w[1] << 16), w[2] | (w[3] << 16), w[4] | (w[5] << 16),
                           w[6] | (w[7] << 16));
        }
    }
}

template <int FP8>
__global__ void __launch_bounds__(kTmaPackThreads, 1)
    pack_tma_kernel(const __grid_constant__ CUtensorMap in_map, long long C, long long S,
                    void* __restrict__ out, const unsigned int* amax_bits, float* scale_out,
                    long long c_tiles, long long s_tiles, long long tiles, int stages, int* status,
                    unsigned long long wait_ns) {
    using Shape = TmaPackShape<FP8>;
    griddep_launch_dependents();   // the conv reading this output waits for completion
    extern __shared__ unsigned char pack_smem[];
    const uint32_t raw = smem_u32(pack_smem);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t full0 = base + static_cast<uint32_t>(stages) * Shape::kStageBytes;
    const uint32_t empty0 = full0 + 8u * stages;
    volatile uint32_t* abort_flag =
        reinterpret_cast<volatile uint32_t*>(pack_smem + (empty0 + 8u * stages - raw));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, kTmaPackConvWarps);
        }
        *abort_flag = 0u;
        fence_mbar_init();
        prefetch_tmap(&in_map);
    }
    // e4m3: quotients by the scale through its reciprocal and one correction
    // step, except for tiny scales or an all-ones significand (IEEE division)
    float scale = 1.0f, rscale = 1.0f;
    bool corr = false;
    if (FP8) {
        scale = fp8_scale_of(amax_bits);
        rscale = __frcp_rn(scale);
        corr = quot_corrected_ok(scale);
        if (blockIdx.x == 0 && threadIdx.x == 0) *scale_out = scale;
    }
    __syncthreads();   // the barriers are initialised before any thread uses them
    long long issued = 0;
    if (warp == kTmaPackConvWarps) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (long long t = blockIdx.x; t < tiles; t += gridDim.x) {
                if (!pack_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag, status, wait_ns)) break;
                const long long ct = t % c_tiles, rest = t / c_tiles;
                const long long st = rest % s_tiles, n = rest / s_tiles;
                mbar_arrive_expect_tx(full0 + 8 * stage, Shape::kStageBytes);
                tma_load_3d(base + stage * Shape::kStageBytes, &in_map, full0 + 8 * stage,
                            static_cast<int>(st * kTmaPackPos), static_cast<int>(ct * Shape::kC),
                            static_cast<int>(n));
                ++issued;
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else {
        // ------------------------------------------------------ converters
        // quarter-warp = 8 consecutive 8-position blocks of one 8-channel group
        const int pb = (warp & 3) * 8 + (lane & 7);          // position block, 0..31
        const int cg = (warp >> 2) * 4 + (lane >> 3);        // channel group, 0..15
        int stage = 0;
        uint32_t phase = 0;
        for (long long t = blockIdx.x; t < tiles; t += gridDim.x) {
            if (!pack_wait(full0 + 8 * stage, phase, abort_flag, status, wait_ns)) break;
            const long long ct = t % c_tiles, rest = t / c_tiles;
            const long long st = rest % s_tiles, n = rest / s_tiles;
            const long long s0 = st * kTmaPackPos + pb * 8;
            const unsigned char* tile = pack_smem + (base - raw) + stage * Shape::kStageBytes;
            {
                const long long c = ct * Shape::kC + cg * 8;
                uint4 v[8];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    v[k] = *reinterpret_cast<const uint4*>(tile + (cg * 8 + k) * (kTmaPackPos * 2) +
                                                            pb * 16);
                if (c < C) {
                    if (corr)
                        pack_unit_store<FP8, true>(v, n, s0, c, C, S, out, scale, rscale);
                    else
                        pack_unit_store<FP8, false>(v, n, s0, c, C, S, out, scale, rscale);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * stage);
            if (++stage == stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    __syncthreads();
    if (*abort_flag && warp == kTmaPackConvWarps && lane == 0) {
        // boxes issued but never waited for land before the CTA leaves
        for (long long i = issued > stages ? issued - stages : 0; i < issued; ++i) {
            const uint32_t bar = full0 + 8 * static_cast<uint32_t>(i % stages);
            const long long t0 = clock64();
            while (!mbar_try_wait(bar, static_cast<uint32_t>((i / stages) & 1)) &&
                   clock64() - t0 < static_cast<long long>(kPackDrainCycles)) {
            }
        }
    }
}

// ----------------------------------------------------------------- row repack
// dst[r, 0:src_row_bytes) = src[r, :], dst[r, src_row_bytes:dst_row_bytes) = 0,
// for two matrices in one launch (the point-output GEMM's A and B operands),
// matrix 1's rows optionally shifted right by shift1 words (zeros in front).
// Gives operands whose rows are not 16-byte aligned a copy the TMA can tile.
// Rows move in W-byte words (W = 8 when both pitches allow, else 4).  Each
// warp copies two rows at a time in spans of 256 words: all loads of both
// rows' span are issued before any store, so a lane keeps up to 16 loads in
// flight.  The kernel lets a dependent launch start early (the GEMM it feeds
// waits for this grid's completion before reading).
template <typename Word>
__global__ void __launch_bounds__(256) row_repack_kernel(const Word* __restrict__ src0,
                                                         Word* __restrict__ dst0, long long rows0,
                                                         const Word* __restrict__ src1,
                                                         Word* __restrict__ dst1, long long rows1,
                                                         long long src_words, long long dst_words,
                                                         long long shift1) {
    griddep_launch_dependents();
    constexpr int kPer = 8;   // words per lane per row and span
    const int lane = threadIdx.x & 31;
    const long long total = rows0 + rows1;
    const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const long long warp = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    for (long long r0 = 2 * warp; r0 < total; r0 += 2 * nwarps) {
        const Word* src[2];
        Word* dst[2];
        bool live[2];
        long long sh[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            long long r = r0 + h;
            live[h] = r < total;
            if (r >= rows0) {
                r -= rows0;
                src[h] = src1 + r * src_words;
                dst[h] = dst1 + r * dst_words;
                sh[h] = shift1;
            } else {
                src[h] = src0 + r * src_words;
                dst[h] = dst0 + r * dst_words;
                sh[h] = 0;
            }
        }
        for (long long base = 0; base < dst_words; base += 32 * kPer) {
            Word v[2][kPer];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const long long w = base + lane + 32 * i - sh[h];   // source word
                    v[h][i] = (live[h] && w >= 0 && w < src_words) ? __ldg(src[h] + w) : Word(0);
                }
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const long long w = base + lane + 32 * i;
                    if (live[h] && w < dst_words) dst[h][w] = v[h][i];
                }
        }
    }
}

// ----------------------------------------------------------------- transpose
// dst[c, r] = src[r, c] for a dense [R, C] 16-bit matrix, into rows of P >= R
// elements whose tail [R, P) is zero-filled (the backward passes of the
// point-output GEMM turn their operands K-major this way).  64x64 tiles
// through shared memory (2-element pitch padding keeps the transposed reads
// free of bank conflicts).  With C and P even, every global access moves an
// element pair (a warp: 128 bytes of a row); otherwise single elements.
__global__ void __launch_bounds__(256) transpose_pad_pairs_kernel(
    const unsigned short* __restrict__ src, long long R, long long C,
    unsigned short* __restrict__ dst, long long P, long long tiles_r, long long tiles_c) {
    griddep_launch_dependents();
    __shared__ __align__(4) unsigned short t[64][66];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (long long b = blockIdx.x; b < tiles_r * tiles_c; b += gridDim.x) {
        const long long r0 = (b % tiles_r) * 64, c0 = (b / tiles_r) * 64;
        const long long c = c0 + 2 * tx;   // this lane's source column pair
        for (int i = ty; i < 64; i += 8) {
            const long long r = r0 + i;
            uint32_t v = 0;
            if (r < R && c < C) v = __ldg(reinterpret_cast<const uint32_t*>(src + r * C + c));
            *reinterpret_cast<uint32_t*>(&t[i][2 * tx]) = v;
        }
        __syncthreads();
        const long long r = r0 + 2 * tx;   // this lane's destination column pair
        for (int i = ty; i < 64; i += 8) {
            const long long cc = c0 + i;
            if (cc < C && r < P) {
                const uint32_t v = static_cast<uint32_t>(t[2 * tx][i]) |
                                   (static_cast<uint32_t>(t[2 * tx + 1][i]) << 16);
                *reinterpret_cast<uint32_t*>(dst + cc * P + r) = v;
            }
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(256) transpose_pad_kernel(const unsigned short* __restrict__ src,
                                                            long long R, long long C,
                                                            unsigned short* __restrict__ dst,
                                                            long long P, long long tiles_r,
                                                            long long tiles_c) {
    griddep_launch_dependents();
    __shared__ unsigned short t[64][66];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (long long b = blockIdx.x; b < tiles_r * tiles_c; b += gridDim.x) {
        const long long r0 = (b % tiles_r) * 64, c0 = (b / tiles_r) * 64;
        for (int i = ty; i < 64; i += 8) {
            const long long r = r0 + i;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const long long c = c0 + 32 * h + tx;
                t[i][32 * h + tx] = (r < R && c < C) ? __ldg(src + r * C + c) : 0;
            }
        }
        __syncthreads();
        for (int i = ty; i < 64; i += 8) {
            const long long c = c0 + i;
            if (c < C) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const long long r = r0 + 32 * h + tx;
                    if (r < P) dst[c * P + r] = t[32 * h + tx][i];
                }
            }
        }
        __syncthreads();
    }
}

// ----------------------------------------------------------------- patch gather
// Convolutions whose stride equals the filter (zero padding): the patches do
// not overlap, and GEMM row m = (n, od, oh, ow) is the patch
// x[n, od*T .. +T, oh*R .. +R, ow*S .. +S, :]: T*R segments of S*C contiguous
// elements.  Each row is written to `a` with a pitch of `pitch` words, its
// tail zeroed; one warp per row.  The lanes walk the row's words 32 apart,
// stepping their (segment, offset) position without divisions, and keep 8
// loads in flight before storing.  Counts are in Word units (a Word holds
// one or more elements; segments and rows are whole Words).
template <typename Word>
__device__ __forceinline__ Word zero_word() {
    Word z;
    memset(&z, 0, sizeof z);
    return z;
}

template <typename Word>
__global__ void __launch_bounds__(256) patch_gather_kernel(
    const Word* __restrict__ x, Word* __restrict__ a, long long M, long long D, long long H,
    long long Wrow, long long seg, int T, int R, int Do, int Ho, int Wo, long long pitch) {
    griddep_launch_dependents();
    constexpr int kBatch = 8;
    const int lane = threadIdx.x & 31;
    const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const long long row_words = static_cast<long long>(T) * R * seg;
    const long long wrap = (H - R + 1) * Wrow;   // from segment (t, R-1) to (t+1, 0)
    for (long long m = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         m < M; m += nwarps) {
        const long long ow = m % Wo;
        long long q = m / Wo;
        const long long oh = q % Ho;
        q /= Ho;
        const long long od = q % Do;
        const long long n = q / Do;
        Word* dst = a + m * pitch;
        // this lane's position: segment base pointer and offset within it
        const Word* sb = x + ((n * D + od * T) * H + oh * R) * Wrow + ow * seg;
        long long off = lane;
        int r = 0;
        auto normalise = [&]() {
            while (off >= seg) {
                off -= seg;
                if (++r == R) {
                    r = 0;
                    sb += wrap;
                } else {
                    sb += Wrow;
                }
            }
        };
        normalise();
        for (long long i = lane; i < row_words; i += 32 * kBatch) {
            const Word* src[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                src[u] = sb + off;
                off += 32;
                normalise();
            }
            Word v[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                v[u] = (i + 32 * u < row_words) ? __ldg(src[u]) : zero_word<Word>();
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (i + 32 * u < row_words) dst[i + 32 * u] = v[u];
        }
        for (long long i = row_words + lane; i < pitch; i += 32) dst[i] = zero_word<Word>();
    }
}

// The same gather with one thread per output word (problems whose word
// counts fit in 32 bits): word w of `a` is row m = w / pitch, word i of it;
// i < T*R*seg reads segment (t, r) = divmod(i / seg, R) at offset i % seg of
// patch (n, od, oh, ow), the rest is the zero tail.  The indices come from
// multiply-shift divisors set on the host (FastDiv), so a thread spends a few
// instructions per 16-byte word; consecutive threads store consecutive
// words (whole rows per warp instruction) and read the patch's contiguous
// S*C-element segments.
struct GatherFlat {
    FastDiv f_pitch, f_seg, f_r, f_wo, f_ho, f_do;
    uint32_t total, row_words, T, R, H, D, Wrow, seg;
};

// One 16-byte word of the gathered rows (output word w, the rows' pitch
// in 16-byte words), assembled from P = 16 / sizeof(In) pieces of the
// patch: piece i of a row is element run `off` of segment sid = (t, r), the
// pieces past the row's T*R*S*C elements zero.  In is the widest piece the
// segments' alignment allows (16, 4, 2 or 1 bytes).
template <typename In>
__device__ __forceinline__ void gather_word(const In* __restrict__ x, uint4* __restrict__ a,
                                            const GatherFlat& g, uint32_t w) {
    constexpr int P = 16 / static_cast<int>(sizeof(In));
    const uint32_t m = fdiv(w, g.f_pitch);
    const uint32_t i0 = (w - m * g.f_pitch.d) * P;   // first piece of this word
    const uint32_t q1 = fdiv(m, g.f_wo), ow = m - q1 * g.f_wo.d;
    const uint32_t q2 = fdiv(q1, g.f_ho), oh = q1 - q2 * g.f_ho.d;
    const uint32_t n = fdiv(q2, g.f_do), od = q2 - n * g.f_do.d;
    uint32_t sid = fdiv(i0, g.f_seg), off = i0 - sid * g.seg;
    union {
        uint4 v;
        In p[P];
    } u;
#pragma unroll
    for (int k = 0; k < P; ++k) {
        if (i0 + k < g.row_words) {
            const uint32_t t = fdiv(sid, g.f_r), r = sid - t * g.R;
            const uint32_t plane = (n * g.D + od * g.T + t) * g.H + oh * g.R + r;
            u.p[k] = __ldg(x + static_cast<size_t>(plane) * g.Wrow + ow * g.seg + off);
        } else {
            u.p[k] = zero_word<In>();
        }
        if (++off == g.seg) {
            off = 0;
            ++sid;
        }
    }
    a[w] = u.v;
}

// One thread per 16-byte word of the gathered rows; a second job (g1.total
// > 0: the weights' rows, copied to the same pitch) takes the words after
// the first job's, so both run in one launch.
template <typename In>
__global__ void __launch_bounds__(256) patch_gather_flat_kernel(const In* __restrict__ x,
                                                                uint4* __restrict__ a, GatherFlat g,
                                                                const In* __restrict__ x1,
                                                                uint4* __restrict__ a1,
                                                                GatherFlat g1) {
    griddep_launch_dependents();
    const uint32_t step = gridDim.x * blockDim.x;
    const uint32_t total = g.total + g1.total;   // below 2^31 (host check)
    for (uint32_t w = blockIdx.x * blockDim.x + threadIdx.x; w < total; w += step) {
        if (w < g.total)
            gather_word(x, a, g, w);
        else
            gather_word(x1, a1, g1, w - g.total);
    }
}

// The geometry of one gather job: rows (n, od, oh, ow) of T*R*S*C elements
// of x, each at `pitch_bytes`, in words of wb bytes.
struct GatherJob {
    long long N, D, H, W, C;
    int T, R, S, Do, Ho, Wo;
    long long seg_b, row_b, M;
};

GatherJob gather_job(int elt, long long N, long long D, long long H, long long W, long long C,
                     int T, int R, int S, int Do, int Ho, int Wo) {
    GatherJob j{N, D, H, W, C, T, R, S, Do, Ho, Wo, 0, 0, 0};
    j.seg_b = static_cast<long long>(S) * C * elt;
    j.row_b = W * C * elt;
    j.M = N * Do * Ho * Wo;
    return j;
}

bool word_fits(const GatherJob& j, long long pitch_bytes, int wb) {
    return j.seg_b % wb == 0 && j.row_b % wb == 0 && pitch_bytes % wb == 0;
}

GatherFlat flat_params(const GatherJob& j, long long pitch_bytes, int wb) {
    GatherFlat g;
    g.total = static_cast<uint32_t>(j.M * (pitch_bytes / 16));
    g.seg = static_cast<uint32_t>(j.seg_b / wb);
    g.row_words = static_cast<uint32_t>(static_cast<long long>(j.T) * j.R * g.seg);
    g.T = static_cast<uint32_t>(j.T);
    g.R = static_cast<uint32_t>(j.R);
    g.H = static_cast<uint32_t>(j.H);
    g.D = static_cast<uint32_t>(j.D);
    g.Wrow = static_cast<uint32_t>(j.row_b / wb);
    g.f_pitch = make_fastdiv(static_cast<uint32_t>(pitch_bytes / 16));
    g.f_seg = make_fastdiv(g.seg);
    g.f_r = make_fastdiv(g.R);
    g.f_wo = make_fastdiv(static_cast<uint32_t>(j.Wo));
    g.f_ho = make_fastdiv(static_cast<uint32_t>(j.Ho));
    g.f_do = make_fastdiv(static_cast<uint32_t>(j.Do));
    return g;
}

// Pieces of the job's rows and of its x against the flat kernel's 32-bit
// indices (the 16-byte output words of the two jobs of one launch together
// below 2^31), and a pitch of whole 16-byte words.
bool flat_ok(const GatherJob& j, long long pitch_bytes, int wb) {
    const long long pieces = j.M * (pitch_bytes / wb);
    const long long x_words = j.N * j.D * j.H * (j.row_b / wb);
    return pitch_bytes % 16 == 0 && pieces > 0 && pieces < (1ll << 31) &&
           x_words < (1ll << 31) && word_fits(j, pitch_bytes, wb);
}

template <typename In>
cudaError_t flat_launch(const void* x, void* a, const GatherFlat& g, const void* x1, void* a1,
                        const GatherFlat& g1, int num_sms, cudaStream_t stream) {
    long long blk = (static_cast<long long>(g.total) + g1.total + 255) / 256;
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (blk > cap) blk = cap;
    const unsigned grid = static_cast<unsigned>(blk < 1 ? 1 : blk);
    patch_gather_flat_kernel<In><<<grid, 256, 0, stream>>>(
        static_cast<const In*>(x), static_cast<uint4*>(a), g, static_cast<const In*>(x1),
        static_cast<uint4*>(a1), g1);
    return cudaGetLastError();
}

// A warp per row (word counts past 32 bits).
cudaError_t row_launch(const void* x, int elt, const GatherJob& j, void* a, long long pitch_bytes,
                       int num_sms, cudaStream_t stream) {
    long long blocks = (j.M + 7) / 8;
    const long long cap = static_cast<long long>(num_sms) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const unsigned grid = static_cast<unsigned>(blocks);
    if (word_fits(j, pitch_bytes, 16))
        patch_gather_kernel<uint4><<<grid, 256, 0, stream>>>(
            static_cast<const uint4*>(x), static_cast<uint4*>(a), j.M, j.D, j.H, j.row_b / 16,
            j.seg_b / 16, j.T, j.R, j.Do, j.Ho, j.Wo, pitch_bytes / 16);
    else if (word_fits(j, pitch_bytes, 4))
        patch_gather_kernel<uint32_t><<<grid, 256, 0, stream>>>(
            static_cast<const uint32_t*>(x), static_cast<uint32_t*>(a), j.M, j.D, j.H,
            j.row_b / 4, j.seg_b / 4, j.T, j.R, j.Do, j.Ho, j.Wo, pitch_bytes / 4);
    else if (elt == 2)
        patch_gather_kernel<unsigned short><<<grid, 256, 0, stream>>>(
            static_cast<const unsigned short*>(x), static_cast<unsigned short*>(a), j.M, j.D, j.H,
            j.row_b / 2, j.seg_b / 2, j.T, j.R, j.Do, j.Ho, j.Wo, pitch_bytes / 2);
    else
        patch_gather_kernel<unsigned char><<<grid, 256, 0, stream>>>(
            static_cast<const unsigned char*>(x), static_cast<unsigned char*>(a), j.M, j.D, j.H,
            j.row_b, j.seg_b, j.T, j.R, j.Do, j.Ho, j.Wo, pitch_bytes);
    return cudaGetLastError();
}

// How the patches (and, with_w, the weights) are gathered: the word width,
// whether the patches take the one-thread-per-word kernel, and whether the
// weights share its launch.
struct GatherPlan {
    GatherJob jx, jw;
    int wb;
    bool flat_x, together;
};

GatherPlan gather_plan(int elt, long long N, long long D, long long H, long long W, long long C,
                       int T, int R, int S, int Do, int Ho, int Wo, long long pitch_bytes,
                       bool with_w, long long K) {
    GatherPlan gp;
    gp.jx = gather_job(elt, N, D, H, W, C, T, R, S, Do, Ho, Wo);
    // the weights: K rows of T*R*S*C elements, each one "patch"
    gp.jw = gather_job(elt, K, 1, 1, 1, static_cast<long long>(T) * R * S * C, 1, 1, 1, 1, 1, 1);
    // one thread per 16-byte output word when every index fits in 32 bits,
    // read in 16-, 4-, 2- or 1-byte pieces: the widest that divides the
    // segment, row and pitch bytes (of both jobs when they share the launch)
    auto widest = [&](bool both) {
        for (int cand : {16, 4})
            if (word_fits(gp.jx, pitch_bytes, cand) && (!both || word_fits(gp.jw, pitch_bytes, cand)))
                return cand;
        return elt;
    };
    // the weights share the launch when that keeps the patches' word width
    gp.wb = widest(false);
    gp.flat_x = flat_ok(gp.jx, pitch_bytes, gp.wb);
    gp.together = with_w && K > 0 && gp.flat_x && widest(true) == gp.wb &&
                  flat_ok(gp.jw, pitch_bytes, gp.wb) &&
                  (gp.jx.M + gp.jw.M) * (pitch_bytes / 16) < (1ll << 31);
    return gp;
}

}  // namespace

int patch_gather_launches(int elt, long long N, long long D, long long H, long long W, long long C,
                          int T, int R, int S, int Do, int Ho, int Wo, long long pitch_bytes,
                          bool with_w, long long K) {
    const GatherPlan gp = gather_plan(elt, N, D, H, W, C, T, R, S, Do, Ho, Wo, pitch_bytes, with_w, K);
    return (with_w && K > 0 && !gp.together) ? 2 : 1;
}

cudaError_t launch_patch_gather(const void* x, int elt, long long N, long long D, long long H,
                                long long W, long long C, int T, int R, int S, int Do, int Ho,
                                int Wo, void* a, long long pitch_bytes, const void* w,
                                long long K, void* wc, int num_sms, cudaStream_t stream) {
    const bool two = w != nullptr && K > 0;
    const GatherPlan gp = gather_plan(elt, N, D, H, W, C, T, R, S, Do, Ho, Wo, pitch_bytes, two, K);
    const GatherJob& jx = gp.jx;
    const GatherJob& jw = gp.jw;
    const int wb = gp.wb;
    const bool flat_x = gp.flat_x, together = gp.together;
    if (flat_x) {
        const GatherFlat gx = flat_params(jx, pitch_bytes, wb);
        GatherFlat gw{};
        if (together) gw = flat_params(jw, pitch_bytes, wb);
        cudaError_t e;
        if (wb == 16)
            e = flat_launch<uint4>(x, a, gx, w, wc, gw, num_sms, stream);
        else if (wb == 4)
            e = flat_launch<uint32_t>(x, a, gx, w, wc, gw, num_sms, stream);
        else if (wb == 2)
            e = flat_launch<unsigned short>(x, a, gx, w, wc, gw, num_sms, stream);
        else
            e = flat_launch<unsigned char>(x, a, gx, w, wc, gw, num_sms, stream);
        if (e != cudaSuccess || !two || together) return e;
    } else {
        cudaError_t e = row_launch(x, elt, jx, a, pitch_bytes, num_sms, stream);
        if (e != cudaSuccess || !two) return e;
    }
    // the weights in a launch of their own
    return launch_patch_gather(w, elt, K, 1, 1, 1, static_cast<long long>(T) * R * S * C, 1, 1, 1,
                               1, 1, 1, wc, pitch_bytes, nullptr, 0, nullptr, num_sms, stream);
}

cudaError_t launch_transpose_pad(const void* src, long long R, long long C, void* dst,
                                 long long P, int num_sms, cudaStream_t stream) {
    if (P < R || R <= 0 || C <= 0) return cudaErrorInvalidValue;
    const long long tiles_r = (P + 63) / 64, tiles_c = (C + 63) / 64;
    long long blocks = tiles_r * tiles_c;
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (C % 2 == 0 && P % 2 == 0) {
        transpose_pad_pairs_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
            static_cast<const unsigned short*>(src), R, C, static_cast<unsigned short*>(dst), P,
            tiles_r, tiles_c);
        return cudaGetLastError();
    }
    transpose_pad_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const unsigned short*>(src), R, C, static_cast<unsigned short*>(dst), P,
        tiles_r, tiles_c);
    return cudaGetLastError();
}

cudaError_t launch_row_repack(const void* src0, void* dst0, long long rows0, const void* src1,
                              void* dst1, long long rows1, long long src_row_bytes,
                              long long dst_row_bytes, long long dst1_shift_bytes, int num_sms,
                              cudaStream_t stream) {
    if (src_row_bytes % 4 || dst_row_bytes % 4 || dst1_shift_bytes % 4 || dst1_shift_bytes < 0 ||
        dst_row_bytes < src_row_bytes + dst1_shift_bytes)
        return cudaErrorInvalidValue;
    const int wb =
        (src_row_bytes % 8 == 0 && dst_row_bytes % 8 == 0 && dst1_shift_bytes % 8 == 0) ? 8 : 4;
    const long long dst_words = dst_row_bytes / wb;
    // two rows per warp, 8 warps per block; at most 4 blocks per SM so that
    // the dependent GEMM's CTAs find room as soon as they are launched
    long long blocks = (rows0 + rows1 + 15) / 16;
    const long long cap = static_cast<long long>(num_sms) * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (wb == 8)
        row_repack_kernel<unsigned long long><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
            static_cast<const unsigned long long*>(src0), static_cast<unsigned long long*>(dst0),
            rows0, static_cast<const unsigned long long*>(src1),
            static_cast<unsigned long long*>(dst1), rows1, src_row_bytes / 8, dst_words,
            dst1_shift_bytes / 8);
    else
        row_repack_kernel<uint32_t><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
            static_cast<const uint32_t*>(src0), static_cast<uint32_t*>(dst0), rows0,
            static_cast<const uint32_t*>(src1), static_cast<uint32_t*>(dst1), rows1,
            src_row_bytes / 4, dst_words, dst1_shift_bytes / 4);
    return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(const float* ws, void* out, long long MK, int splits,
                                 const float* scale_x, const float* scale_w, const float* bias,
                                 long long K, int act, int num_sms, cudaStream_t stream) {
    const long long units = (MK & 3) == 0 ? (MK >> 2) : MK;
    long long blocks = (units + 255) / 256;
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    splitk_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        ws, reinterpret_cast<__nv_bfloat16*>(out), MK, splits, scale_x, scale_w, bias, K, act);
    return cudaGetLastError();
}

cudaError_t launch_amax_bf16(const void* in, long long n, unsigned int* amax_bits, int num_sms,
                             cudaStream_t stream) {
    long long blocks = (n / 8 + 255) / 256;
    const long long cap = static_cast<long long>(num_sms) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    amax_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        reinterpret_cast<const __nv_bfloat16*>(in), n, amax_bits);
    return cudaGetLastError();
}

int pack_tma_stages(int fp8, int smem_optin) {
    const uint32_t sb = fp8 ? TmaPackShape<1>::kStageBytes : TmaPackShape<0>::kStageBytes;
    const int fit = static_cast<int>((static_cast<long long>(smem_optin) - 1024 - 256) / sb);
    return fit < 2 ? 0 : (fit > 8 ? 8 : fit);
}

cudaError_t launch_pack_tma(const CUtensorMap* in_map, long long N, long long C, long long S,
                            void* out, int fp8, const unsigned int* amax_bits, float* scale_out,
                            int num_sms, int smem_optin, int* status, unsigned long long wait_ns,
                            cudaStream_t stream) {
    const int stages = pack_tma_stages(fp8, smem_optin);
    if (stages < 2 || C % 8 || S % 8) return cudaErrorInvalidValue;
    const long long tc = fp8 ? TmaPackShape<1>::kC : TmaPackShape<0>::kC;
    const long long c_tiles = (C + tc - 1) / tc;
    const long long s_tiles = (S + kTmaPackPos - 1) / kTmaPackPos;
    const long long tiles = N * c_tiles * s_tiles;
    const long long grid = tiles < num_sms ? tiles : num_sms;
    const uint32_t sb = fp8 ? TmaPackShape<1>::kStageBytes : TmaPackShape<0>::kStageBytes;
    const size_t smem = 1024 + static_cast<size_t>(stages) * sb + 16u * stages + 16;
    cudaError_t e;
    static std::atomic<int> smem_set[2][kMaxDevices];
    if (fp8) {
        e = ensure_dynamic_smem(pack_tma_kernel<1>, smem, smem_set[1]);
        if (e != cudaSuccess) return e;
        pack_tma_kernel<1><<<static_cast<unsigned>(grid), kTmaPackThreads, smem, stream>>>(
            *in_map, C, S, out, amax_bits, scale_out, c_tiles, s_tiles, tiles, stages, status,
            wait_ns);
    } else {
        e = ensure_dynamic_smem(pack_tma_kernel<0>, smem, smem_set[0]);
        if (e != cudaSuccess) return e;
        pack_tma_kernel<0><<<static_cast<unsigned>(grid), kTmaPackThreads, smem, stream>>>(
            *in_map, C, S, out, amax_bits, scale_out, c_tiles, s_tiles, tiles, stages, status,
            wait_ns);
    }
    return cudaGetLastError();
}

cudaError_t launch_pack(const void* in, long long N, long long C, long long S, void* out, int fp8,
                        const unsigned int* amax_bits, float* scale_out, int num_sms,
                        cudaStream_t stream) {
    const auto* x = reinterpret_cast<const __nv_bfloat16*>(in);
    if (C % 16 == 0 && S % 8 == 0) {
        // warp tile: 32 channels x 128 positions for e4m3 output (each
        // channel row read 256 bytes at a time; measured 1.63 against 1.68 ms
        // for amax + pack of the 3.5 GB fp8 workload activation), 64 x 64
        // for bf16 output (1.17 against 1.39 ms); the pack_lanes override sets it
        int lc = fp8 ? 2 : 4;
        const int lanes = overrides().pack_lanes;
        if (lanes == 2 || lanes == 4) lc = lanes;
        const long long c_tiles = (C + 16 * lc - 1) / (16 * lc);
        const long long s_tiles = (S + 256 / lc - 1) / (256 / lc);
        const long long tiles = N * c_tiles * s_tiles;   // one warp per tile
        long long blocks = (tiles + 7) / 8;
        const long long cap = static_cast<long long>(num_sms) * 8;
        if (blocks > cap) blocks = cap;
        const unsigned nb = static_cast<unsigned>(blocks);
        if (fp8 && lc == 2)
            pack_tiles_kernel<1, 2><<<nb, 256, 0, stream>>>(x, C, S, out, amax_bits, scale_out,
                                                            c_tiles, s_tiles, tiles);
        else if (fp8)
            pack_tiles_kernel<1, 4><<<nb, 256, 0, stream>>>(x, C, S, out, amax_bits, scale_out,
                                                            c_tiles, s_tiles, tiles);
        else if (lc == 2)
            pack_tiles_kernel<0, 2><<<nb, 256, 0, stream>>>(x, C, S, out, amax_bits, scale_out,
                                                            c_tiles, s_tiles, tiles);
        else
            pack_tiles_kernel<0, 4><<<nb, 256, 0, stream>>>(x, C, S, out, amax_bits, scale_out,
                                                            c_tiles, s_tiles, tiles);
        return cudaGetLastError();
    }
    const long long c_tiles = (C + kPackC - 1) / kPackC;
    const long long s_tiles = (S + kPackS - 1) / kPackS;
    const long long blocks = N * c_tiles * s_tiles;
    if (blocks <= 0 || blocks > 0x7FFFFFFFll) return cudaErrorInvalidValue;
    if (fp8)
        pack_kernel<1><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
            x, N, C, S, out, amax_bits, scale_out, c_tiles, s_tiles);
    else
        pack_kernel<0><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
            x, N, C, S, out, amax_bits, scale_out, c_tiles, s_tiles);
    return cudaGetLastError();
}

}  // namespace c3d
