// conv_fused_q.cu -- e4m3 forward convolution of a bf16 channel-major (NCDHW)
// activation, quantised while the A operand is built: no NCDHW -> NDHWC pack
// pass.  This is the NCDHW-direct loader FlyDSL PR #860 leaves to future work
// in its 3x1x1 unfold-revert commit (a kernel reading NCDHW straight into the
// GEMM without materialising A), in its e4m3 form: the codes are exactly the
// pack's, e4m3_satfinite_rn(x / scale) with scale = amax / 448 (the tiled
// bf16 -> fp8 pack commit), so the result is the conv of the packed tensor.
//
// Filters T = 1, R x S with "same" padding (ph = (R-1)/2, pw = (S-1)/2),
// unit stride and dilation: each output frame reads one input frame.
//
// Output rows run over padded rows: per frame, P = h * Wp + wp, Wp = W + 2pw,
// image column w = wp - pw.  A CTA's 128 rows [P0, P0 + 128) read, for tap
// (r, s), the input at padded position P + (r - ph) * Wp + (s - pw): the
// same 128 rows of one strip of L padded positions starting at
// P0 - ph * Wp - pw, shifted by r * Wp + s.  The strip holds zeros at the
// padding columns and outside the frame, so every tap is exact, and the
// tensor core reads each tap's A operand in place through a shared-memory
// descriptor whose start address moves by (r * Wp + s) * 16 bytes.  The strip
// is stored K-major without swizzle: 8 slices of 16 channels (one per 16-byte
// core-matrix column), each slice L rows of 16 bytes (SBO 128 bytes between
// 8-row groups, LBO L * 16 bytes between slices).  Each input element is
// converted about L / 128 times (2.5 for a 3x3 filter on a 90-wide frame)
// instead of once per tap, and rows with wp outside the image (2 of every
// Wp) are computed and dropped.
//
// Warp roles (480 threads):
//   warp 0      TMA producer of the e4m3 KTRSC weight: per chunk and group of
//               tap_group consecutive taps one box of 128 channel bytes x
//               (BN >> pair) filters x tap_group taps, 128-byte swizzle, into
//               a ring (full / empty mbarriers);
//   warp 1      TMEM allocation; lane 0 issues tcgen05.mma kind::f8f6f4
//               (cta_group::2 for CTA pairs): per weight stage the four MMAs
//               of each of its taps, then one commit;
//   warps 2..5  epilogue: tcgen05.ld -> scale_x * scale_w (+ bias) -> bf16 ->
//               16-byte stores of the valid rows; overlaps the next unit;
//   warp 6      strip loader (with a scratch): copies each converted strip
//               back from this CTA's scratch for every column tile;
//   warps 7..14 converters: warp k builds slice k (16 channels) of a chunk's
//               strip -- one m-tile ahead into the scratch through a staging
//               buffer when there is one, else in place in a strip buffer --:
//               each lane takes 8 consecutive image positions of the frame
//               rows the strip covers, loads them from the 16 channel planes
//               (16-byte loads, 512 contiguous bytes of a plane per warp),
//               quantises them to e4m3 and writes each position's 16 channel
//               bytes to its strip row; strip rows with no image position are
//               zeroed.
// Every wait is bounded; on expiry the kernel records CONV_ERR_TIMEOUT,
// drains its copies and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>

#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace c3d {

namespace {

constexpr int kFqConvWarps = 8;    // one per 16-channel slice of a 128-channel chunk
constexpr int kFqEpiWarp0 = 2;
constexpr int kFqLoaderWarp = 6;
constexpr int kFqConvWarp0 = 7;
constexpr int kFqChunk = 128;      // channels (e4m3 bytes) per reduction chunk

struct FqUnit {
    int frame, mt, nt;
};

// The i-th unit of the CTA (pair) whose m-tiles are g0, g0 + gs, ...: every
// column tile of one m-tile in turn, then the next m-tile, so the strips
// converted for the first column tile serve the others.  False past the end.
__device__ __forceinline__ bool fq_unit(int i, int g0, int gs, const FQParams& p, FqUnit& r) {
    const int k = i / p.n_tiles;
    const int g = g0 + k * gs;
    if (g >= p.m_tiles) return false;
    r.nt = i - k * p.n_tiles;
    r.frame = g / p.mt_frame;
    r.mt = g - r.frame * p.mt_frame;
    return true;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ int floor_div(int a, int b) {
    const int q = a / b;
    return (a % b != 0 && ((a < 0) != (b < 0))) ? q - 1 : q;
}

// store_row_bf16 with streaming (evict-first) stores: the output is written
// once and never read here, so it should not push the scratch out of L2.
__device__ __forceinline__ void store_row_bf16_stream(__nv_bfloat16* dst, const uint32_t (&v)[32],
                                                      float scale, const float* bias, int count,
                                                      bool vec_ok) {
    auto val = [&](int i) {
        return __uint_as_float(v[i]) * scale + (bias ? __ldg(bias + i) : 0.0f);
    };
    if (count == 32 && vec_ok) {
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            __stcs(d4 + i, make_uint4(pack_bf16x2(val(8 * i + 0), val(8 * i + 1)),
                                      pack_bf16x2(val(8 * i + 2), val(8 * i + 3)),
                                      pack_bf16x2(val(8 * i + 4), val(8 * i + 5)),
                                      pack_bf16x2(val(8 * i + 6), val(8 * i + 7))));
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < count) dst[i] = __float2bfloat16_rn(val(i));
    }
}

// Columns the unit's MMAs compute: BN, or the rest of K rounded up to 32.
__device__ __forceinline__ int fq_cols(int nt, const FQParams& p) {
    const int rest = p.K - nt * p.BN;
    return rest >= p.BN ? p.BN : ((rest + 31) & ~31);
}

// One 16-channel slice (channels c0 .. c0+15) of a strip, converted to e4m3
// in the shared-memory rows at dst0 (L rows of 16 bytes): strip row q holds
// padded position Ps + q of frame (n, d); rows with no image position are
// zeros.  Run by one warp.
__device__ __forceinline__ void fq_convert_slice(const FQParams& p, uint32_t dst0, int c0, int Ps,
                                                 int n, int d, int lane, float scale_x,
                                                 float rscale, bool corr) {
    const long long HW = static_cast<long long>(p.H) * p.W;
    const bool vec_planes = (HW % 8) == 0;   // every channel plane 16-byte aligned
    const int nch = min(16, p.C - c0);
    // (1) strip rows that hold no image position (padding columns,
    // rows outside the frame, or channels past C) are zeros
    {
        int h = floor_div(Ps + lane, p.Wp);
        int wp = Ps + lane - h * p.Wp;
        for (int qb = 0; qb < p.L; qb += 32) {
            const int w = wp - p.pw;
            if (!(h >= 0 && h < p.H && w >= 0 && w < p.W) || nch <= 0)
                st_shared_v4(dst0 + static_cast<uint32_t>(qb + lane) * 16u, 0u, 0u, 0u,
                             0u);
            wp += 32;
            while (wp >= p.Wp) {
                wp -= p.Wp;
                ++h;
            }
        }
    }
    // (2) the image rows the strip covers, 8 positions x 16
    // channels per lane: one 16-byte load per channel plane (a
    // warp reads 512 contiguous bytes of each), the 8 x 16
    // transpose in registers, one 16-byte strip row per position.
    // Needs 16-byte aligned planes (H*W % 8 == 0); otherwise (3).
    if (nch > 0 && vec_planes) {
        const int ha = max(0, floor_div(Ps, p.Wp));
        const int hb = min(p.H - 1, floor_div(Ps + p.L - 1, p.Wp));
        const long long fa = static_cast<long long>(ha) * p.W;
        const long long fb = static_cast<long long>(hb + 1) * p.W;
        const unsigned short* src0 =
            p.x + ((static_cast<long long>(n) * p.C + c0) * p.D + d) * HW;
        const long long cstride = static_cast<long long>(p.D) * HW;
        for (long long f = (fa & ~7ll) + 8 * lane; f < fb; f += 256) {
            // codes[e][j]: channels 4j .. 4j+3 of position f + e
            uint32_t codes[8][4];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint4 v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int c = 8 * half + i;
                    v[i] = c < nch
                               ? __ldcs(reinterpret_cast<const uint4*>(src0 + c * cstride + f))
                               : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    // element e of each channel row: word e/2, low or high half
                    float xv[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t ww = (e >> 1) == 0 ? v[i].x : (e >> 1) == 1 ? v[i].y
                                          : (e >> 1) == 2 ? v[i].z : v[i].w;
                        xv[i] = __uint_as_float((e & 1) ? (ww & 0xFFFF0000u) : (ww << 16));
                    }
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float* x4 = xv + 4 * j;
                        codes[e][2 * half + j] =
                            corr ? (quant_e4m3x2<true>(x4[0], x4[1], scale_x, rscale) |
                                    (quant_e4m3x2<true>(x4[2], x4[3], scale_x, rscale) << 16))
                                 : (quant_e4m3x2<false>(x4[0], x4[1], scale_x, rscale) |
                                    (quant_e4m3x2<false>(x4[2], x4[3], scale_x, rscale) << 16));
                    }
                }
            }
            int h = static_cast<int>(f / p.W);
            int w = static_cast<int>(f - static_cast<long long>(h) * p.W);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int q = h * p.Wp + w + p.pw - Ps;
                if (f + e >= fa && f + e < fb && q >= 0 && q < p.L)
                    st_shared_v4(dst0 + static_cast<uint32_t>(q) * 16u, codes[e][0],
                                 codes[e][1], codes[e][2], codes[e][3]);
                if (++w == p.W) {
                    w = 0;
                    ++h;
                }
            }
        }
    }
    // (3) planes not 16-byte aligned: per strip row, 16 2-byte
    // loads (lanes take consecutive rows, so a warp reads 64
    // contiguous bytes of a plane per load)
    if (nch > 0 && !vec_planes) {
        const unsigned short* src0 =
            p.x + ((static_cast<long long>(n) * p.C + c0) * p.D + d) * HW;
        const long long cstride = static_cast<long long>(p.D) * HW;
        int h = floor_div(Ps + lane, p.Wp);
        int wp = Ps + lane - h * p.Wp;
        for (int qb = 0; qb < p.L; qb += 32) {
            const int w = wp - p.pw;
            if (h >= 0 && h < p.H && w >= 0 && w < p.W) {
                const unsigned short* src = src0 + static_cast<long long>(h) * p.W + w;
                float xv[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    xv[i] = __uint_as_float(
                        (i < nch ? static_cast<uint32_t>(__ldg(src + i * cstride)) : 0u) << 16);
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    o[j] = corr ? (quant_e4m3x2<true>(xv[4 * j], xv[4 * j + 1], scale_x, rscale) |
                                   (quant_e4m3x2<true>(xv[4 * j + 2], xv[4 * j + 3], scale_x,
                                                       rscale) << 16))
                                : (quant_e4m3x2<false>(xv[4 * j], xv[4 * j + 1], scale_x, rscale) |
                                   (quant_e4m3x2<false>(xv[4 * j + 2], xv[4 * j + 3], scale_x,
                                                        rscale) << 16));
                st_shared_v4(dst0 + static_cast<uint32_t>(qb + lane) * 16u, o[0], o[1],
                             o[2], o[3]);
            }
            wp += 32;
            while (wp >= p.Wp) {
                wp -= p.Wp;
                ++h;
            }
        }
    }
}

template <int PAIR>
__global__ void __launch_bounds__(kFqThreads, 1)
    conv_fused_q_kernel(const __grid_constant__ CUtensorMap w_map, const FQParams p) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t strips = base;                                     // 2 strip buffers
    const uint32_t staging = base + ((2u * p.strip_bytes + 1023u) & ~1023u);   // converters' rows
    const uint32_t ring = staging + ((p.strip_bytes + 1023u) & ~1023u);
    const uint32_t bfull0 = ring + static_cast<uint32_t>(p.b_stages) * p.b_stage_bytes;
    const uint32_t bempty0 = bfull0 + 8u * p.b_stages;
    const uint32_t sfull0 = bempty0 + 8u * p.b_stages;
    const uint32_t sempty0 = sfull0 + 16u;
    const uint32_t tfull0 = sempty0 + 16u;
    const uint32_t tempty0 = tfull0 + 16u;
    const uint32_t kready0 = tempty0 + 16u;   // ahead mode: scratch slot written / copied out
    const uint32_t kfree0 = kready0 + 16u;
    const uint32_t drain_bar = kfree0 + 16u;
    const uint32_t lbar0 = drain_bar + 8u;   // the loader's strip copies
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem_raw + (lbar0 + 8u - raw));
    // misc[0] TMEM base, misc[1] abort flag, misc[2] weight boxes issued, misc[3] consumed
    volatile uint32_t* abort_flag = misc + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    // ahead mode: the converters work one m-tile ahead into the scratch and a
    // loader copies strips back; otherwise they convert in place
    const bool ahead = p.scratch != nullptr;
    // the scratch strips are read back n_tiles times within about a unit's
    // time: they are asked to outlive the streaming activation and output in L2
    const uint64_t keep_pol = l2_policy_evict_last();
    const int unit0 = static_cast<int>(blockIdx.x) >> PAIR;
    const int ustride = static_cast<int>(gridDim.x) >> PAIR;
    const int taps = p.R * p.S;
    constexpr int kTileM = 128 << PAIR;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.b_stages; ++s) {
            mbar_init(bfull0 + 8 * s, 1);
            mbar_init(bempty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            // a strip is signalled by the loader (ahead mode) or by every
            // converter warp, of both CTAs of a pair
            mbar_init(sfull0 + 8 * b, (ahead ? 1 : kFqConvWarps) * (1 + PAIR));
            mbar_init(sempty0 + 8 * b, 1);
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, kEpiWarps * (1 + PAIR));
            mbar_init(kready0 + 8 * b, kFqConvWarps);
            mbar_init(kfree0 + 8 * b, 1);
        }
        mbar_init(drain_bar, 1);
        mbar_init(lbar0, 1);
        misc[1] = 0u;
        misc[2] = 0u;
        misc[3] = 0u;
        fence_mbar_init();
        prefetch_tmap(&w_map);
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(smem_u32(misc), p.tmem_cols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(misc), p.tmem_cols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();   // both CTAs' barriers exist before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = misc[0];
    // the amax word is written by the kernel before this one in the stream
    const float scale_x = fp8_scale_of(p.amax_bits);
    uint32_t loads = 0;          // converter lane 0: its slice reloads (barrier parity)
    bool load_pending = false;   // converter lane 0: a reload issued and not seen landing

    if (warp == 0) {
        // ------------------------------------------------------ weight producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0;
            bool ok = true;
            FqUnit t;
            for (int i = 0; ok && fq_unit(i, unit0, ustride, p, t); ++i) {
                const int n0 = t.nt * p.BN + static_cast<int>(rank) * (fq_cols(t.nt, p) >> PAIR);
                for (int cc = 0; cc < p.chunks && ok; ++cc) {
                    // one box per group of tap_group consecutive taps
                    for (int tap = 0; tap < taps; tap += p.tap_group) {
                        if (!wait_bar(bempty0 + 8 * stage, phase ^ 1u, abort_flag, p.status,
                                      p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        uint32_t fb = bfull0 + 8 * stage;
                        if (PAIR) {
                            if (rank == 0) mbar_arrive_expect_tx(fb, 2u * p.b_stage_bytes);
                            fb = mapa_shared(fb, 0);
                            tma_load_3d_pair(ring + stage * p.b_stage_bytes, &w_map, fb,
                                             cc * kFqChunk, n0, tap);
                        } else {
                            mbar_arrive_expect_tx(fb, p.b_stage_bytes);
                            tma_load_3d(ring + stage * p.b_stage_bytes, &w_map, fb, cc * kFqChunk,
                                        n0, tap);
                        }
                        misc[2] = ++issued;
                        if (++stage == p.b_stages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0 && rank == 0) {
            // descriptors built once and stepped by encoded offsets (16-byte
            // units): strip buffer, tap window (r * Wp + s rows), two slices
            // per MMA; weight stage, 32 bytes per MMA
            const uint32_t lbo = static_cast<uint32_t>(p.L) * 16u;          // slice stride
            const uint64_t adesc0 = make_smem_desc(strips, 128u, 0u, lbo);   // no swizzle
            const uint64_t bdesc0 = make_smem_desc(ring, 1024u, 2u);         // 128B swizzle
            const uint32_t a_buf_step = p.strip_bytes >> 4;
            const uint32_t a_kstep = (2u * lbo) >> 4;
            const uint32_t b_stage_step = p.b_stage_bytes >> 4;
            const uint32_t b_tap_step = (p.b_stage_bytes / p.tap_group) >> 4;   // one tap's block
            const int row_skip = p.Wp - p.S;   // window offset from (r, S) to (r + 1, 0)
            int stage = 0, acc_iter = 0, chunk_iter = 0;
            uint32_t phase = 0, consumed = 0;
            bool ok = true;
            FqUnit t;
            for (int i = 0; ok && fq_unit(i, unit0, ustride, p, t); ++i) {
                const int acc = acc_iter & 1;
                const uint32_t acc_phase = static_cast<uint32_t>(acc_iter >> 1) & 1u;
                if (!wait_bar(tempty0 + 8 * acc, acc_phase ^ 1u, abort_flag, p.status, p.wait_ns))
                    break;
                tc_fence_after();
                const uint32_t idesc =
                    (p.idesc & ~(0x3Fu << 17)) | (static_cast<uint32_t>(fq_cols(t.nt, p) >> 3) << 17);
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * p.BN);
                uint32_t accum = 0u;
                for (int cc = 0; cc < p.chunks && ok; ++cc, ++chunk_iter) {
                    const int sb = chunk_iter & 1;
                    const uint32_t s_phase = static_cast<uint32_t>(chunk_iter >> 1) & 1u;
                    if (!wait_bar(sfull0 + 8 * sb, s_phase, abort_flag, p.status, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t abuf = adesc0 + static_cast<uint64_t>(sb) * a_buf_step;
                    int win = 0, s = 0;   // window offset of tap (r, s): r * Wp + s
                    for (int tap0 = 0; tap0 < taps; tap0 += p.tap_group) {
                        // one weight stage: tap_group taps (fewer in the last
                        // group of an odd count), each a block of filter rows
                        if (!wait_bar(bfull0 + 8 * stage, phase, abort_flag, p.status, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        misc[3] = ++consumed;
                        const int ntap = min(p.tap_group, taps - tap0);
                        uint64_t b = bdesc0 + static_cast<uint64_t>(stage) * b_stage_step;
                        for (int j = 0; j < ntap; ++j, b += b_tap_step) {
                            const uint64_t a = abuf + static_cast<uint64_t>(win);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {   // 32 channel bytes per MMA
                                if (PAIR)
                                    tc_mma_f8_pair(d_tmem, a + kk * a_kstep, b + 2u * kk, idesc,
                                                   accum);
                                else
                                    tc_mma_f8(d_tmem, a + kk * a_kstep, b + 2u * kk, idesc, accum);
                                accum = 1u;
                            }
                            ++win;
                            if (++s == p.S) {
                                s = 0;
                                win += row_skip;
                            }
                        }
                        if (PAIR)
                            tc_commit_pair(bempty0 + 8 * stage, 3);
                        else
                            tc_commit(bempty0 + 8 * stage);
                        if (++stage == p.b_stages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    // the strip buffer is free in both CTAs once these MMAs have read it
                    if (ok) {
                        if (PAIR)
                            tc_commit_pair(sempty0 + 8 * sb, 3);
                        else
                            tc_commit(sempty0 + 8 * sb);
                    }
                }
                if (!ok) break;
                if (PAIR)
                    tc_commit_pair(tfull0 + 8 * acc, 3);
                else
                    tc_commit(tfull0 + 8 * acc);
                ++acc_iter;
            }
        }
    } else if (warp < kFqEpiWarp0 + kEpiWarps) {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;   // TMEM lane quarter this warp may read
        float scale = scale_x;
        if (p.scale_w) scale *= *p.scale_w;
        if (blockIdx.x == 0 && threadIdx.x == kFqEpiWarp0 * 32 && p.scale_x_out)
            *p.scale_x_out = scale_x;
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
        const bool vec_out = (p.K % 8) == 0;
        const uint32_t tempty_dst0 = PAIR ? mapa_shared(tempty0, 0) : tempty0;
        int acc_iter = 0;
        FqUnit t;
        for (int i = 0; fq_unit(i, unit0, ustride, p, t); ++i) {
            const int acc = acc_iter & 1;
            const uint32_t acc_phase = static_cast<uint32_t>(acc_iter >> 1) & 1u;
            if (!wait_bar(tfull0 + 8 * acc, acc_phase, abort_flag, p.status, p.wait_ns)) break;
            tc_fence_after();
            // this thread's output row: padded position -> image position
            const int P = t.mt * kTileM + static_cast<int>(rank) * 128 + q * 32 + lane;
            const int h = P / p.Wp, wp = P - h * p.Wp;
            const bool valid = P < p.HWp && wp >= p.pw && wp < p.pw + p.W;
            const long long orow =
                (static_cast<long long>(t.frame) * p.H + h) * p.W + (wp - p.pw);
            const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                static_cast<uint32_t>(acc * p.BN);
            const int nch = min(p.BN / 32, (p.K - t.nt * p.BN + 31) / 32);
            for (int j = 0; j < nch; ++j) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tb + 32 * j, v);
                tmem_ld_wait();
                const int n0 = t.nt * p.BN + 32 * j;
                if (valid)
                    store_row_bf16_stream(out + orow * p.K + n0, v, scale,
                                          p.bias ? p.bias + n0 : nullptr, min(32, p.K - n0),
                                          vec_out);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR)
                    mbar_arrive_cluster(tempty_dst0 + 8 * acc);
                else
                    mbar_arrive(tempty0 + 8 * acc);
            }
            ++acc_iter;
        }
    } else if (warp == kFqLoaderWarp) {
        // ------------------------------------------------------ strip loader
        // (ahead mode): each chunk's converted strip comes back from this
        // CTA's scratch slot of the m-tile, one bulk copy into a strip buffer
        if (ahead && lane == 0) {
            const uint32_t sfull_dst0 = PAIR ? mapa_shared(sfull0, 0) : sfull0;
            const unsigned char* mine =
                p.scratch + static_cast<long long>(blockIdx.x) * p.scratch_stride;
            int chunk_iter = 0;
            bool ok = true;
            FqUnit t;
            for (int i = 0; ok && fq_unit(i, unit0, ustride, p, t); ++i) {
                const int j = i / p.n_tiles, slot = j & 1;
                // the converters have written the m-tile's strips
                if (t.nt == 0 && !wait_bar(kready0 + 8 * slot, static_cast<uint32_t>(j >> 1) & 1u,
                                           abort_flag, p.status, p.wait_ns)) {
                    ok = false;
                    break;
                }
                for (int cc = 0; cc < p.chunks; ++cc, ++chunk_iter) {
                    const int sb = chunk_iter & 1;
                    const uint32_t s_phase = static_cast<uint32_t>(chunk_iter >> 1) & 1u;
                    if (!wait_bar(sempty0 + 8 * sb, s_phase ^ 1u, abort_flag, p.status, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(lbar0, p.strip_bytes);
                    bulk_load_1d_hint(strips + static_cast<uint32_t>(sb) * p.strip_bytes,
                                      mine + (static_cast<long long>(slot) * p.chunks + cc) *
                                                 p.strip_bytes,
                                      p.strip_bytes, lbar0, keep_pol);
                    load_pending = true;
                    if (!wait_bar(lbar0, loads & 1u, abort_flag, p.status, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    load_pending = false;
                    ++loads;
                    if (PAIR)
                        mbar_arrive_cluster(sfull_dst0 + 8 * sb);
                    else
                        mbar_arrive(sfull0 + 8 * sb);
                }
                // the slot's last strip has landed: the converters may refill it
                if (ok && t.nt == p.n_tiles - 1) mbar_arrive(kfree0 + 8 * slot);
            }
        }
    } else {
        // ------------------------------------------------------ converters
        const int k = warp - kFqConvWarp0;   // 16-channel slice of each chunk
        const float rscale = __frcp_rn(scale_x);
        const bool corr = quot_corrected_ok(scale_x);
        bool ok = true;
        if (ahead) {
            // one m-tile ahead of the MMAs: m-tile j's strips into scratch
            // slot j & 1, slice by slice through this warp's staging rows
            unsigned char* mine = p.scratch + static_cast<long long>(blockIdx.x) * p.scratch_stride;
            const uint32_t slice_bytes = static_cast<uint32_t>(p.L) * 16u;
            const uint32_t stage = staging + static_cast<uint32_t>(k) * slice_bytes;
            for (int j = 0; ok; ++j) {
                const int g = unit0 + j * ustride;
                if (g >= p.m_tiles) break;
                const int frame = g / p.mt_frame, mt = g - frame * p.mt_frame;
                const int n = frame / p.D, d = frame - n * p.D;
                const int Ps = mt * kTileM + static_cast<int>(rank) * 128 - (p.ph * p.Wp + p.pw);
                const int slot = j & 1;
                // the loader has copied out the slot's previous m-tile
                if (j >= 2 && !wait_bar(kfree0 + 8 * slot, static_cast<uint32_t>((j >> 1) - 1) & 1u,
                                        abort_flag, p.status, p.wait_ns)) {
                    ok = false;
                    break;
                }
                for (int cc = 0; cc < p.chunks; ++cc) {
                    // the staging rows' previous bulk store has read them
                    if (lane == 0) bulk_wait_read<0>();
                    __syncwarp();
                    fq_convert_slice(p, stage, cc * kFqChunk + k * 16, Ps, n, d, lane, scale_x,
                                     rscale, corr);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        bulk_store_1d_hint(mine + ((static_cast<long long>(slot) * p.chunks + cc) *
                                                       kFqConvWarps + k) * slice_bytes,
                                           stage, slice_bytes, keep_pol);
                        bulk_commit();
                    }
                }
                if (lane == 0) {
                    bulk_wait_done<0>();   // the slot's slices are in memory
                    mbar_arrive(kready0 + 8 * slot);
                }
                __syncwarp();
            }
        } else {
            // in place: each chunk's slice straight into a strip buffer
            const uint32_t sfull_dst0 = PAIR ? mapa_shared(sfull0, 0) : sfull0;
            int chunk_iter = 0;
            FqUnit t;
            for (int i = 0; ok && fq_unit(i, unit0, ustride, p, t); ++i) {
                const int n = t.frame / p.D, d = t.frame - n * p.D;
                const int Ps = t.mt * kTileM + static_cast<int>(rank) * 128 - (p.ph * p.Wp + p.pw);
                for (int cc = 0; cc < p.chunks; ++cc, ++chunk_iter) {
                    const int sb = chunk_iter & 1;
                    const uint32_t s_phase = static_cast<uint32_t>(chunk_iter >> 1) & 1u;
                    if (!wait_bar(sempty0 + 8 * sb, s_phase ^ 1u, abort_flag, p.status, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    fq_convert_slice(p,
                                     strips + static_cast<uint32_t>(sb) * p.strip_bytes +
                                         static_cast<uint32_t>(k) * static_cast<uint32_t>(p.L) * 16u,
                                     cc * kFqChunk + k * 16, Ps, n, d, lane, scale_x, rscale, corr);
                    // the strip's generic-proxy writes become visible to the
                    // tensor core before the MMA issuer learns of them
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (PAIR)
                            mbar_arrive_cluster(sfull_dst0 + 8 * sb);
                        else
                            mbar_arrive(sfull0 + 8 * sb);
                    }
                }
            }
        }
    }

    if (ahead && lane == 0) {
        // the converters' bulk stores have read their staging rows (and
        // written) before the CTA leaves; a strip reload that was not seen
        // landing lands first
        if (warp >= kFqConvWarp0) bulk_wait_done<0>();
        if (warp == kFqLoaderWarp && load_pending) drain_wait(lbar0, loads & 1u);
    }
    __syncthreads();
    // in a pair, both CTAs finish their roles (and the peer's last remote
    // arrivals land) before either drains, frees TMEM or leaves
    if (PAIR) cluster_sync();
    if (PAIR && *abort_flag) {
        const long long t0 = clock64();
        while (clock64() - t0 < 200000) {
        }
    }
    if (*abort_flag) {
        // weight boxes armed but never consumed, then the MMAs in flight
        if (warp == 0 && lane == 0 && rank == 0) {
            const uint32_t issued = misc[2], consumed = misc[3];
            for (uint32_t i = consumed; i < issued; ++i)
                drain_wait(bfull0 + 8 * (i % static_cast<uint32_t>(p.b_stages)),
                           (i / static_cast<uint32_t>(p.b_stages)) & 1u);
        }
        if (warp == 1 && lane == 0 && rank == 0) {
            if (PAIR)
                tc_commit_pair(drain_bar, 1);
            else
                tc_commit(drain_bar);
            drain_wait(drain_bar, 0);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        if (PAIR)
            tmem_dealloc_pair(tmem_base, p.tmem_cols);
        else
            tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

template <int PAIR>
cudaError_t launch_fq(const CUtensorMap* w_map, const FQParams& p, int grid, size_t smem,
                      cudaStream_t stream) {
    auto kern = conv_fused_q_kernel<PAIR>;
    static std::atomic<int> smem_set[kMaxDevices];
    cudaError_t e = ensure_dynamic_smem(kern, smem, smem_set);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kFqThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    int n = 0;
    if (PAIR) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 2;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, *w_map, p);
}

}  // namespace

cudaError_t launch_fused_q(const CUtensorMap* w_map, const FQParams& p, int grid, size_t smem,
                           cudaStream_t stream) {
    return p.pair ? launch_fq<1>(w_map, p, grid, smem, stream)
                  : launch_fq<0>(w_map, p, grid, smem, stream);
}

}  // namespace c3d
