// conv_igemm.cu -- the forward implicit-GEMM convolution kernel for sm_103a.
//
// GEMM view (FlyDSL PR #860 "fp8 conv3d: 8-wave GEMM pipeline + BIG_IN fix",
// PR summary): rows M = output positions (n, od, oh, ow), columns = the K
// filters, reduction over (channel chunk, tap) of the KTRSC weight rows.  A
// point-output conv is the same kernel with a plain row-major A (MIOpen PR
// #10912, description).
//
// One persistent CTA per SM (or CTA pair per two SMs) walks a strided list of
// work units (m-tile, n-tile, split) of one launch's m-tile range.  Warp roles:
//   warp 0      TMA producer: the A and B boxes of each k-step (one or two
//               128-byte boxes per operand, per row sub-tile) into a
//               multi-stage shared-memory ring (full/empty mbarriers).  The A
//               box is an im2col-mode box (generic conv), a 4-D tiled box of
//               H*W rows (T x 1 x 1 temporal conv) or a 2-D tiled box (GEMM:
//               K-major, MN-major, or one of two row phases); padding taps
//               and reduction tails read as zeros through TMA bounds.
//   warp 1      allocates TMEM; lane 0 issues tcgen05.mma (kind::f16 for
//               bf16, kind::f8f6f4 for e4m3; cta_group::2 for pairs) into
//               fp32 accumulators and commits stages back to the producer.
//   warps 2..5  epilogue: tcgen05.ld -> scale (+ bias) -> bf16 -> staged in
//               shared memory -> TMA tensor stores, or 8- / 4-byte stores for
//               rows that are not 16-byte multiples, or direct fp32 split-K
//               partials; overlaps the next unit's mainloop.
//   warps 6..9  (row-gather GEMM only) cp.async producers for operands whose
//               rows are not 16-byte aligned and no workspace is given.
// Every wait is bounded: on expiry the kernel records CONV_ERR_TIMEOUT,
// drains its copies and MMAs in flight, frees TMEM and returns.
#include <cuda_bf16.h>

#include <type_traits>

#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace c3d {

namespace {


struct Unit {
    int m_tile, n_tile, split;
};

// Columns unit t's MMAs compute: BN, or for a last column tile that K does
// not fill, the rest of K rounded up to 32 (whole 32-column epilogue chunks;
// a tcgen05 N for either CTA count).
__device__ __forceinline__ int tile_cols(int n_tile, const KParams& p) {
    const int rest = p.K - n_tile * p.BN;
    return rest >= p.BN ? p.BN : ((rest + 31) & ~31);
}

// Temporal m-tile -> ((n, d) plane, H*W tile).  Plane-major by default (output
// row order); H*W-tile-major when p.hw_major, so that the units running at
// once cover one H*W tile of consecutive planes and share their input planes
// (each is read by T output planes) in L2.
__device__ __forceinline__ void temporal_tile(int m_tile, const KParams& p, int& plane, int& hwb) {
    if (p.hw_major) {
        hwb = static_cast<int>(fdiv(static_cast<uint32_t>(m_tile), p.f_planes));
        plane = m_tile - hwb * p.N * p.Do;
    } else {
        plane = static_cast<int>(fdiv(static_cast<uint32_t>(m_tile), p.f_hw_tiles));
        hwb = m_tile - plane * p.hw_tiles;
    }
}

// Work unit -> (m-tile, n-tile, split).  Within a split, tiles are walked in
// groups of `group_m` m-tiles: down M first, then across N, so that CTAs
// running at the same time share both A rows and B columns in L2.  A launch
// covers the m-tiles [m_tile0, m_tile0 + m_tiles) and the column tiles
// [n_tile0, n_tile0 + n_tiles).
__device__ __forceinline__ Unit decode_unit(int u, const KParams& p) {
    const int tiles = p.m_tiles * p.n_tiles;
    Unit r;
    r.split = static_cast<int>(fdiv(static_cast<uint32_t>(u), p.f_tiles));
    const int t = u - r.split * tiles;
    const int group = p.group_m * p.n_tiles;
    const int g = static_cast<int>(fdiv(static_cast<uint32_t>(t), p.f_group));
    const int first_m = g * p.group_m;
    const int gm = min(p.group_m, p.m_tiles - first_m);   // the last group may be short
    const int local = t - g * group;
    const int col = gm == p.group_m ? static_cast<int>(fdiv(static_cast<uint32_t>(local), p.f_gm))
                                    : local / gm;
    r.m_tile = p.m_tile0 + first_m + (local - col * gm);
    r.n_tile = p.n_tile0 + col;
    return r;
}

__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
    uint2 r;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(addr) : "memory");
    return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// The same with an activation after the bias: act(v * scale + bias).  Plans
// with an activation store through this path only; it is kept out of line so
// that its code (one loop per activation) stays out of the kernel's body.
__device__ __noinline__ void store_row_bf16_act(__nv_bfloat16* dst, const uint32_t (&v)[32],
                                                float scale, const float* bias, int act,
                                                int count, bool vec_ok) {
    float y[32];
#pragma unroll
    for (int i = 0; i < 32; ++i)
        y[i] = __uint_as_float(v[i]) * scale + (bias && i < count ? __ldg(bias + i) : 0.0f);
    if (act == kActRelu) {
#pragma unroll
        for (int i = 0; i < 32; ++i) y[i] = activate_c<kActRelu>(y[i]);
    } else if (act == kActSilu) {
#pragma unroll
        for (int i = 0; i < 32; ++i) y[i] = activate_c<kActSilu>(y[i]);
    } else if (act == kActGelu) {
#pragma unroll
        for (int i = 0; i < 32; ++i) y[i] = activate_c<kActGelu>(y[i]);
    }
    if (count == 32 && vec_ok) {
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            d4[i] = make_uint4(pack_bf16x2(y[8 * i + 0], y[8 * i + 1]),
                               pack_bf16x2(y[8 * i + 2], y[8 * i + 3]),
                               pack_bf16x2(y[8 * i + 4], y[8 * i + 5]),
                               pack_bf16x2(y[8 * i + 6], y[8 * i + 7]));
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < count) dst[i] = __float2bfloat16_rn(y[i]);
    }
}

// Store 32 fp32 split-K partial columns of one output row.
__device__ __forceinline__ void store_row_f32(float* dst, const uint32_t (&v)[32], int count,
                                              bool vec_ok) {
    if (count == 32 && vec_ok) {
        float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            d4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < count) dst[i] = __uint_as_float(v[i]);
    }
}

// L2 prefetch of rows [r0, r1) of a row-major matrix with row_bytes per row;
// the byte range is trimmed inward to 16-byte boundaries (the allocation
// starts 16-byte aligned), so it never leaves the matrix.
__device__ __forceinline__ void prefetch_rows(const unsigned char* base, long long r0, long long r1,
                                              long long row_bytes) {
    if (r1 <= r0) return;
    const long long lo = ((r0 * row_bytes) + 15) & ~15ll;
    const long long hi = (r1 * row_bytes) & ~15ll;
    for (long long a = lo; a < hi; a += 65536) {
        const long long n = min(65536ll, hi - a);
        prefetch_l2_bulk(base + a, static_cast<uint32_t>(n));
    }
}

// cp.async row-gather producer (AM_GEMM_GATHER): 128 threads copy the A and B
// tiles of each k-step (128-byte rows) in VEC-byte pieces into the
// 128B-swizzled layout, zero filling rows past M / K and columns past the
// reduction length.  Each thread owns one piece position and every RPP-th
// row, so per piece it only steps a source pointer and a destination offset.
// A stage is released LAG k-steps after its copies were issued, so LAG
// k-steps of copies stay in flight per thread.
template <int VEC, int LAG>
__device__ void gather_producer(const KParams& p, uint32_t tiles, uint32_t full0, uint32_t empty0,
                                volatile uint32_t* abort_flag, int g) {
    constexpr int PPR = 128 / VEC;                 // pieces per 128-byte row
    constexpr int RPP = kGatherThreads / PPR;      // rows covered per pass
    const int total_units = p.m_tiles * p.n_tiles * p.splits;
    const int row0 = g / PPR;
    const int byte = (g % PPR) * VEC;
    const int chunk = byte >> 4, lo = byte & 15;
    const long long rb = p.g_row_bytes;
    int stage = 0;
    uint32_t phase = 0;
    long long it = 0;
    bool ok_run = true;
    for (int u = blockIdx.x; u < total_units && ok_run; u += gridDim.x) {
        const Unit t = decode_unit(u, p);
        const int ks0 = t.split * p.steps_per_split;
        const int ks1 = min(p.k_steps, ks0 + p.steps_per_split);
        const long long m0 = static_cast<long long>(t.m_tile) * kBM + row0;
        const long long n0 = static_cast<long long>(t.n_tile) * p.BN + row0;
        for (int ks = ks0; ks < ks1; ++ks) {
            if (!wait_bar(empty0 + 8 * stage, phase ^ 1u, abort_flag, p.status, p.wait_ns)) {
                ok_run = false;
                break;
            }
            const uint32_t adst = tiles + stage * p.stage_bytes;
            const uint32_t bdst = adst + p.a_stage_bytes;
            const long long colb = static_cast<long long>(ks) * 128 + byte;
            const bool col_ok = colb < rb;
            {
                const unsigned char* src = p.ga + m0 * rb + colb;
                long long m = m0;
#pragma unroll 4
                for (int row = row0; row < kBM; row += RPP) {
                    const bool ok = col_ok && m < p.M;
                    const uint32_t dst = adst + row * 128 + (((chunk ^ (row & 7)) << 4) | lo);
                    cp_async<VEC>(dst, ok ? src : p.ga, ok ? VEC : 0u);
                    src += RPP * rb;
                    m += RPP;
                }
            }
            {
                const unsigned char* src = p.gb + n0 * rb + colb;
                long long n = n0;
#pragma unroll 4
                for (int row = row0; row < p.BN; row += RPP) {
                    const bool ok = col_ok && n < p.K;
                    const uint32_t dst = bdst + row * 128 + (((chunk ^ (row & 7)) << 4) | lo);
                    cp_async<VEC>(dst, ok ? src : p.gb, ok ? VEC : 0u);
                    src += RPP * rb;
                    n += RPP;
                }
            }
            cp_async_commit();
            if (it >= LAG) {
                cp_async_wait<LAG>();
                fence_proxy_async_smem();
                mbar_arrive(full0 + 8 * static_cast<uint32_t>((it - LAG) % p.stages));
            }
            ++it;
            if (++stage == p.stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    cp_async_wait_all();
    fence_proxy_async_smem();
    if (ok_run && !*abort_flag) {
        for (long long j = (it > LAG ? it - LAG : 0); j < it; ++j)
            mbar_arrive(full0 + 8 * static_cast<uint32_t>(j % p.stages));
    }
}

// The MMA issuer (one thread): per k-step, wait for the stage, issue KMMA
// tcgen05.mma over its 32-byte K slices into the tile's TMEM accumulator, and
// commit the stage back to the producer; per tile, commit the accumulator to
// the epilogue.  Shared-memory descriptors are built once and advanced by
// adding encoded byte offsets (address field = bytes >> 4).  A 256-byte
// k-step (KMMA = 8) holds each operand as two 128-byte-swizzled boxes, one
// after the other; slices 4..7 read the second box.
//
// The tensor pipe queues only a couple of MMAs, so an issue blocks until the
// pipe has room and the issuer runs in step with it: whatever the thread does
// between two k-steps (the barrier wait, the commit, the loop) must fit in the
// MMAs still queued, or the pipe idles.  With two or more slices per k-step
// the next k-step's stage is therefore tested (without blocking) before the
// last slice is issued, while the earlier slices are still executing: when it
// has landed, the next k-step starts without a wait.  A stage still in flight
// is waited for as usual after the commit (blocking there instead would hold
// back this stage's release to the producer).  At the last k-step of a unit
// the same slot decodes the next unit and tests its accumulator.
template <int KMMA, int FP8, int PAIR, int MSUB>
__device__ __forceinline__ void mma_issuer(const KParams& p, uint32_t tiles, uint32_t full0,
                                           uint32_t empty0, uint32_t tfull0, uint32_t tempty0,
                                           uint32_t tmem_base, uint32_t* misc,
                                           volatile uint32_t* abort_flag) {
    const int total_units = p.m_tiles * p.n_tiles * p.splits;
    // MN-major A (SW128): 64-element MN blocks 8 KB apart (two per 128-row
    // tile), 8-row K groups 1 KB apart; a 16-row K slice advances 2 KB
    const uint64_t adesc0 = p.a_mn ? make_smem_desc(tiles, 1024u, p.layout, 8192u)
                                   : make_smem_desc(tiles, p.sbo, p.layout);
    const uint32_t a_slice = p.a_mn ? 128u : 2u;   // encoded advance per 16-element K slice
    const uint64_t bdesc0 = make_smem_desc(tiles + p.a_stage_bytes, p.sbo, p.layout);
    const uint32_t stage_step = p.stage_bytes >> 4;
    // msub row sub-tiles share each B stage; the TMEM holds 2/msub unit
    // accumulators (double-buffered when msub == 1)
    constexpr int nacc = 2 / MSUB;
    constexpr bool kEarly = KMMA >= 2;
    const uint32_t sub_step = (static_cast<uint32_t>(kBM) * p.BK) >> 4;   // A sub-tile, encoded
    const uint32_t abox_step = (static_cast<uint32_t>(kBM) * 128u) >> 4;
    const uint32_t bbox_step = (static_cast<uint32_t>(p.BN >> PAIR) * 128u) >> 4;
    const int ustride = static_cast<int>(gridDim.x) >> PAIR;
    int u = static_cast<int>(blockIdx.x) >> PAIR;
    if (u >= total_units) return;
    Unit t = decode_unit(u, p);
    int stage = 0, acc_iter = 0;
    uint32_t phase = 0, consumed = 0;
    bool stage_ready = false;   // the full barrier of `stage` was already waited for
    bool acc_ready = false;     // the accumulator of `acc_iter` was already waited for
    while (true) {
        const int ks0 = t.split * p.steps_per_split;
        const int ks1 = min(p.k_steps, ks0 + p.steps_per_split);
        const int acc = acc_iter % nacc;
        if (!acc_ready) {
            const uint32_t acc_phase = static_cast<uint32_t>(acc_iter / nacc) & 1u;
            if (!wait_bar(tempty0 + 8 * acc, acc_phase ^ 1u, abort_flag, p.status, p.wait_ns)) return;
            tc_fence_after();
        }
        acc_ready = false;
        // the instruction descriptor's N (bits 17-22, N / 8) for this tile
        const uint32_t idesc = (p.idesc & ~(0x3Fu << 17)) |
                               (static_cast<uint32_t>(tile_cols(t.n_tile, p) >> 3) << 17);
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * MSUB * p.BN);
        const int un = u + ustride;
        Unit tn = t;
        uint32_t accum = 0u;
        for (int ks = ks0; ks < ks1; ++ks) {
            if (!stage_ready) {
                if (!wait_bar(full0 + 8 * stage, phase, abort_flag, p.status, p.wait_ns)) return;
                misc[3] = ++consumed;
                tc_fence_after();
            }
            stage_ready = false;
            int nstage = stage + 1;
            uint32_t nphase = phase;
            if (nstage == p.stages) {
                nstage = 0;
                nphase ^= 1u;
            }
            const uint64_t off = static_cast<uint64_t>(static_cast<uint32_t>(stage) * stage_step);
            const uint64_t ad = adesc0 + off, bd = bdesc0 + off;
#pragma unroll
            for (int k = 0; k < KMMA; ++k) {
                if (kEarly && k == KMMA - 1) {
                    const bool last = ks + 1 == ks1;
                    if (!last || un < total_units) {
                        if (last) {
                            tn = decode_unit(un, p);
                            if (nacc == 2) {
                                const int na = acc_iter + 1;
                                const uint32_t na_phase = static_cast<uint32_t>(na / nacc) & 1u;
                                acc_ready = mbar_test_wait(tempty0 + 8 * (na % nacc), na_phase ^ 1u);
                            }
                        }
                        if (mbar_test_wait(full0 + 8 * nstage, nphase)) {
                            misc[3] = ++consumed;
                            stage_ready = true;
                        }
                        if (stage_ready || acc_ready) tc_fence_after();
                    }
                }
                const int box = k >> 2, kin = k & 3;   // 128-byte box, 32-byte slice in it
                const uint64_t b = bd + box * bbox_step + 2 * kin;
#pragma unroll
                for (int sub = 0; sub < MSUB; ++sub) {
                    const uint32_t d = d_tmem + static_cast<uint32_t>(sub * p.BN);
                    const uint64_t a = ad + sub * sub_step + box * abox_step + a_slice * kin;
                    if (PAIR) {
                        if (FP8)
                            tc_mma_f8_pair(d, a, b, idesc, accum);
                        else
                            tc_mma_f16_pair(d, a, b, idesc, accum);
                    } else {
                        if (FP8)
                            tc_mma_f8(d, a, b, idesc, accum);
                        else
                            tc_mma_f16(d, a, b, idesc, accum);
                    }
                }
                accum = 1u;
            }
            // the stage is free in both CTAs once these MMAs have read it
            if (PAIR)
                tc_commit_pair(empty0 + 8 * stage, 3);
            else
                tc_commit(empty0 + 8 * stage);
            stage = nstage;
            phase = nphase;
        }
        if (PAIR)
            tc_commit_pair(tfull0 + 8 * acc, 3);
        else
            tc_commit(tfull0 + 8 * acc);
        ++acc_iter;
        if (un >= total_units) break;
        u = un;
        t = kEarly ? tn : decode_unit(un, p);
    }
}

// The TMA producer (one thread): per k-step, wait for a free stage, arm its
// full barrier with the stage's bytes (both CTAs' in a pair) and issue the A
// boxes of each of the MSUB row sub-tiles and the B boxes: NB boxes of
// 128-byte rows per operand for a 256-byte k-step, else one.
template <int AMODE, int FP8, int PAIR, int MSUB, int NB>
__device__ __forceinline__ void tma_producer(const TMaps& tm, const KParams& p, uint32_t tiles,
                                             uint32_t full0,
                                             uint32_t empty0, uint32_t* misc,
                                             volatile uint32_t* abort_flag, uint32_t rank) {
    constexpr int kTileM = kBM << PAIR;
    constexpr int kElt = FP8 ? 1 : 2;
    const int bke = p.BK / kElt;
    const int box_e = bke / NB;                                    // elements per box row
    const uint32_t abox = static_cast<uint32_t>(kBM) * (p.BK / NB);            // A box bytes
    const uint32_t bbox = static_cast<uint32_t>(p.BN >> PAIR) * (p.BK / NB);   // B box bytes
    const int total_units = p.m_tiles * p.n_tiles * p.splits;
    const int unit0 = static_cast<int>(blockIdx.x) >> PAIR;
    const int ustride = static_cast<int>(gridDim.x) >> PAIR;
    int stage = 0;
    uint32_t phase = 0, issued = 0;
    bool ok_run = true;
    for (int u = unit0; u < total_units && ok_run; u += ustride) {
        const Unit t = decode_unit(u, p);
        const int ks0 = t.split * p.steps_per_split;
        const int ks1 = min(p.k_steps, ks0 + p.steps_per_split);
        // row phase (two-phase point-output GEMM): its own A / B maps, local m-tile
        const int rphase = t.m_tile >= p.mt_phase0 ? 1 : 0;
        const int mt_local = t.m_tile - rphase * p.mt_phase0;
        const CUtensorMap* tmA = &tm.a[rphase];
        const CUtensorMap* tmB = &tm.b[rphase];
        // this CTA's B rows: all BN columns, or its half of them in a pair
        // (a pair splits the tile's MMA columns evenly: the peer's half starts
        // at half of this tile's computed width)
        const int n0 = t.n_tile * p.BN + static_cast<int>(rank) * (tile_cols(t.n_tile, p) >> PAIR);
        // A coordinates of each row sub-tile (128 rows of this CTA)
        int aw[2] = {0, 0}, ah[2] = {0, 0}, ad[2] = {0, 0}, an[2] = {0, 0}, am0[2] = {0, 0};
        for (int sub = 0; sub < MSUB; ++sub) {
            const int first = sub * kTileM + kBM * static_cast<int>(rank);
            if (AMODE == AM_IM2COL) {
                const long long m0 =
                    static_cast<long long>(t.m_tile) * kTileM * MSUB + first;
                int ow, oh, od;
                if (p.rows32) {
                    const uint32_t x = static_cast<uint32_t>(m0);
                    const uint32_t q1 = fdiv(x, p.f_Wo);
                    const uint32_t q2 = fdiv(q1, p.f_Ho);
                    const uint32_t q3 = fdiv(q2, p.f_Do);
                    ow = static_cast<int>(x - q1 * static_cast<uint32_t>(p.Wo));
                    oh = static_cast<int>(q1 - q2 * static_cast<uint32_t>(p.Ho));
                    od = static_cast<int>(q2 - q3 * static_cast<uint32_t>(p.Do));
                    an[sub] = static_cast<int>(q3);
                } else {
                    ow = static_cast<int>(m0 % p.Wo);
                    const long long q1 = m0 / p.Wo;
                    oh = static_cast<int>(q1 % p.Ho);
                    const long long q2 = q1 / p.Ho;
                    od = static_cast<int>(q2 % p.Do);
                    an[sub] = static_cast<int>(q2 / p.Do);
                }
                aw[sub] = ow * p.sw - p.pw;
                ah[sub] = oh * p.sh - p.ph;
                ad[sub] = od * p.sd - p.pd;
            } else if (AMODE == AM_TEMPORAL) {
                int plane, hwb;
                temporal_tile(t.m_tile, p, plane, hwb);
                const int nn = static_cast<int>(fdiv(static_cast<uint32_t>(plane), p.f_Do));
                const int od = plane - nn * p.Do;
                an[sub] = nn;
                ad[sub] = od * p.sd - p.pd;
                ah[sub] = hwb * kTileM * MSUB + first;   // first H*W row
            } else {
                am0[sub] = mt_local * kTileM * MSUB + first;
            }
        }
        // reduction order: channel chunk (outer), tap (t, r, s) inner.  The
        // position is decoded once per unit and then stepped incrementally.
        int tap = 0, c0 = 0, fs = 0, fr = 0, ft = 0;
        if (ks0 > 0) {
            const int chunk = static_cast<int>(fdiv(static_cast<uint32_t>(ks0), p.f_taps));
            tap = ks0 - chunk * p.taps;
            c0 = chunk * bke;
            const int qs = static_cast<int>(fdiv(static_cast<uint32_t>(tap), p.f_S));
            ft = static_cast<int>(fdiv(static_cast<uint32_t>(qs), p.f_R));
            fs = tap - qs * p.S;
            fr = qs - ft * p.R;
        }
        int k0 = ks0 * bke;   // GEMM modes: first reduction element of the k-step
        for (int ks = ks0; ks < ks1; ++ks) {
            if (!wait_bar(empty0 + 8 * stage, phase ^ 1u, abort_flag, p.status, p.wait_ns)) {
                ok_run = false;
                break;
            }
            uint32_t fb = full0 + 8 * stage;
            if (PAIR) {
                // the leader's full barrier counts both CTAs' bytes
                if (rank == 0) mbar_arrive_expect_tx(fb, 2u * p.stage_bytes);
                fb = mapa_shared(fb, 0);
            } else {
                mbar_arrive_expect_tx(fb, p.stage_bytes);
            }
            const uint32_t adst0 = tiles + stage * p.stage_bytes;
            const uint32_t bdst = adst0 + p.a_stage_bytes;
            if (AMODE == AM_GEMM_TMA) {
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    const int kj = k0 + j * box_e;
                    for (int sub = 0; sub < MSUB; ++sub) {
                        const uint32_t adst = adst0 + (sub * NB + j) * abox;
                        if (p.a_mn) {
                            // MN-major A: two boxes of 64 MN x 64 K rows
                            if (PAIR) {
                                tma_load_2d_pair(adst, tmA, fb, am0[sub], kj);
                                tma_load_2d_pair(adst + 8192u, tmA, fb, am0[sub] + 64, kj);
                            } else {
                                tma_load_2d(adst, tmA, fb, am0[sub], kj);
                                tma_load_2d(adst + 8192u, tmA, fb, am0[sub] + 64, kj);
                            }
                        } else if (PAIR) {
                            tma_load_2d_pair(adst, tmA, fb, kj, am0[sub]);
                        } else {
                            tma_load_2d(adst, tmA, fb, kj, am0[sub]);
                        }
                    }
                    if (PAIR)
                        tma_load_2d_pair(bdst + j * bbox, tmB, fb, kj, n0);
                    else
                        tma_load_2d(bdst + j * bbox, tmB, fb, kj, n0);
                }
                k0 += bke;
            } else {
                const uint16_t ow = static_cast<uint16_t>(fs * p.dw);
                const uint16_t oh = static_cast<uint16_t>(fr * p.dh);
                const uint16_t od = static_cast<uint16_t>(ft * p.dd);
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    const int cj = c0 + j * box_e;   // channels past C read as zeros
                    for (int sub = 0; sub < MSUB; ++sub) {
                        const uint32_t adst = adst0 + (sub * NB + j) * abox;
                        if (AMODE == AM_TEMPORAL && p.a_mn) {
                            // channel-major x (NCDHW): the tap's input plane
                            // as two MN-major boxes of 64 H*W positions x 64
                            // channels (map dims {H*W, D, C, N})
                            const int dpl = ad[sub] + ft * p.dd;
                            if (PAIR) {
                                tma_load_4d_pair(adst, tmA, fb, ah[sub], dpl, cj, an[sub]);
                                tma_load_4d_pair(adst + 8192u, tmA, fb, ah[sub] + 64, dpl, cj,
                                                 an[sub]);
                            } else {
                                tma_load_4d(adst, tmA, fb, ah[sub], dpl, cj, an[sub]);
                                tma_load_4d(adst + 8192u, tmA, fb, ah[sub] + 64, dpl, cj, an[sub]);
                            }
                        } else if (PAIR) {
                            if (AMODE == AM_IM2COL)
                                tma_load_im2col_5d_pair(adst, tmA, fb, cj, aw[sub], ah[sub],
                                                        ad[sub], an[sub], ow, oh, od);
                            else
                                tma_load_4d_pair(adst, tmA, fb, cj, ah[sub], ad[sub] + ft * p.dd,
                                                 an[sub]);
                        } else {
                            if (AMODE == AM_IM2COL)
                                tma_load_im2col_5d(adst, tmA, fb, cj, aw[sub], ah[sub], ad[sub],
                                                   an[sub], ow, oh, od);
                            else
                                tma_load_4d(adst, tmA, fb, cj, ah[sub], ad[sub] + ft * p.dd,
                                            an[sub]);
                        }
                    }
                    if (PAIR)
                        tma_load_3d_pair(bdst + j * bbox, tmB, fb, cj, tap, n0);
                    else
                        tma_load_3d(bdst + j * bbox, tmB, fb, cj, tap, n0);
                }
                ++tap;
                if (++fs == p.S) {
                    fs = 0;
                    if (++fr == p.R) {
                        fr = 0;
                        if (++ft == p.T) {
                            ft = 0;
                            tap = 0;
                            c0 += bke;
                        }
                    }
                }
            }
            misc[2] = ++issued;
            if (++stage == p.stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// PAIR = 1: CTA-pair variant (a cluster of two CTAs on two SMs computes a
// 256-row tile with tcgen05.mma.cta_group::2; each CTA loads its own 128 A
// rows and half of the tile's B rows, the pair's leader issues the MMAs, and
// each CTA's epilogue drains its own TMEM half).
template <int AMODE, int FP8, int PAIR>
__global__ void __launch_bounds__(AMODE == AM_GEMM_GATHER ? 320 : 192, 1)
    conv_igemm_kernel(const __grid_constant__ TMaps tm, const KParams p) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* base_ptr = smem_raw + (base - raw);
    const uint32_t tiles = base;
    const uint32_t ring_bytes = static_cast<uint32_t>(p.stages) * p.stage_bytes;
    const uint32_t epi0 = base + ring_bytes;   // epilogue staging (1024-aligned)
    const uint32_t full0 = epi0 + p.epi_bytes;
    const uint32_t empty0 = full0 + 8u * p.stages;
    const uint32_t tfull0 = empty0 + 8u * p.stages;
    const uint32_t tempty0 = tfull0 + 16u;
    const uint32_t drain_bar = tempty0 + 16u;
    uint32_t* misc =
        reinterpret_cast<uint32_t*>(base_ptr + ring_bytes + p.epi_bytes + 16u * p.stages + 40u);
    // misc[0] TMEM base, misc[1] abort flag, misc[2] k-steps issued, misc[3] k-steps consumed
    volatile uint32_t* abort_flag = misc + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int total_units = p.m_tiles * p.n_tiles * p.splits;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;   // CTA within the pair
    const int unit0 = static_cast<int>(blockIdx.x) >> PAIR;
    const int ustride = static_cast<int>(gridDim.x) >> PAIR;
    constexpr int kTileM = kBM << PAIR;   // rows of a row sub-tile (a unit has msub of them)
    constexpr bool kGather = (AMODE == AM_GEMM_GATHER);

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(full0 + 8 * s, kGather ? kGatherThreads : 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull0 + 8 * a, 1);
            mbar_init(tempty0 + 8 * a, kEpiWarps * (1 + PAIR));
        }
        mbar_init(drain_bar, 1);
        misc[1] = 0u;
        misc[2] = 0u;
        misc[3] = 0u;
        fence_mbar_init();
        if (!kGather) {
            for (int ph = 0; ph < p.phases; ++ph) {
                prefetch_tmap(&tm.a[ph]);
                prefetch_tmap(&tm.b[ph]);
            }
        }
        if (p.epi_mode == 1)
            for (int ph = 0; ph < p.phases; ++ph) prefetch_tmap(&tm.c[ph]);
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
    // everything above touches only shared memory, TMEM and the kernel
    // parameters; global memory is read and written only after the previous
    // kernel in the stream has completed (programmatic dependent launch)
    griddep_wait();

    if (warp == 0) {
        if (kGather && lane == 0) {
            // row-gather GEMM: warm L2 with the rows this CTA gathers, so the
            // cp.async pieces hit L2 instead of DRAM; each A row block is
            // prefetched once (by its first column tile), each B block by the
            // first row tile
            for (int u = blockIdx.x; u < total_units; u += gridDim.x) {
                const Unit t = decode_unit(u, p);
                const long long m0 = static_cast<long long>(t.m_tile) * kBM;
                const long long n0 = static_cast<long long>(t.n_tile) * p.BN;
                if (t.n_tile == p.n_tile0 && t.split == 0)
                    prefetch_rows(p.ga, m0, min(m0 + kBM, p.M), p.g_row_bytes);
                if (t.m_tile == p.m_tile0 && t.split == 0)
                    prefetch_rows(p.gb, n0, min(n0 + p.BN, static_cast<long long>(p.K)),
                                  p.g_row_bytes);
            }
        }
        // ------------------------------------------------------ TMA producer
        if (!kGather && lane == 0) {
#define C3D_PROD(MS, NBX) \
    tma_producer<AMODE, FP8, PAIR, MS, NBX>(tm, p, tiles, full0, empty0, misc, abort_flag, rank)
            if (p.msub == 2) {
                if (p.BK == 256) C3D_PROD(2, 2);
                else C3D_PROD(2, 1);
            } else {
                if (p.BK == 256) C3D_PROD(1, 2);
                else C3D_PROD(1, 1);
            }
#undef C3D_PROD
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0 && rank == 0) {
#define C3D_MMA(KM, MS) \
    mma_issuer<KM, FP8, PAIR, MS>(p, tiles, full0, empty0, tfull0, tempty0, tmem_base, misc, abort_flag)
            if (p.msub == 2) {
                if (p.BK == 256) C3D_MMA(8, 2);
                else if (p.BK == 128) C3D_MMA(4, 2);
                else if (p.BK == 64) C3D_MMA(2, 2);
                else C3D_MMA(1, 2);
            } else {
                if (p.BK == 256) C3D_MMA(8, 1);
                else if (p.BK == 128) C3D_MMA(4, 1);
                else if (p.BK == 64) C3D_MMA(2, 1);
                else C3D_MMA(1, 1);
            }
#undef C3D_MMA
        }
    } else if (warp < 2 + kEpiWarps) {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;   // TMEM lane quarter this warp may read
        float scale = 1.0f;
        if (p.scale_x) scale *= *p.scale_x;
        if (p.scale_w) scale *= *p.scale_w;
        const bool vec_out = (p.K % 8) == 0;
        const bool vec_ws = (p.K % 4) == 0;
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
        const int nacc = 2 / p.msub;
        const int unit_rows = kTileM * p.msub;
        int acc_iter = 0, epi_iter = 0;
        // the MMA issuer waits on the pair leader's accumulator-free barrier
        const uint32_t tempty_dst0 = PAIR ? mapa_shared(tempty0, 0) : tempty0;
        const uint32_t bufs = epi0 + static_cast<uint32_t>(warp - 2) * 2u * kEpiChunkBytes;
        for (int u = unit0; u < total_units; u += ustride) {
            const Unit t = decode_unit(u, p);
            const int acc = acc_iter % nacc;
            const uint32_t acc_phase = static_cast<uint32_t>(acc_iter / nacc) & 1u;
            // this lane's bias entry of each 32-column chunk of the unit
            // (loaded while the accumulator is still being computed)
            float bl[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int col = t.n_tile * p.BN + 32 * j + lane;
                bl[j] = (p.bias && 32 * j < p.BN && col < p.K) ? __ldg(p.bias + col) : 0.0f;
            }
            if (!wait_bar(tfull0 + 8 * acc, acc_phase, abort_flag, p.status, p.wait_ns)) break;
            tc_fence_after();
            int plane = 0, unit_row0;   // temporal: plane and first H*W row of the unit
            const int rphase = t.m_tile >= p.mt_phase0 ? 1 : 0;   // row phase (GEMM)
            const long long phase_rows = rphase ? p.rows1 : p.rows0;
            if (AMODE == AM_TEMPORAL) {
                int hwb;
                temporal_tile(t.m_tile, p, plane, hwb);
                unit_row0 = hwb * unit_rows;
            } else {
                unit_row0 = (t.m_tile - rphase * p.mt_phase0) * unit_rows;
            }
            for (int sub = 0; sub < p.msub; ++sub) {
                // this thread's row of the unit, and the warp's first row
                const int wrow0 = unit_row0 + sub * kTileM + kBM * static_cast<int>(rank) + q * 32;
                const int r = wrow0 + lane;
                long long m;
                bool valid, any;
                if (AMODE == AM_TEMPORAL) {
                    valid = r < p.HW;
                    any = wrow0 < p.HW;
                    m = static_cast<long long>(plane) * p.HW + r;
                } else {
                    valid = r < phase_rows;
                    any = wrow0 < phase_rows;
                    m = static_cast<long long>(r) * p.phases + rphase;   // output row
                }
                const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                    static_cast<uint32_t>((acc * p.msub + sub) * p.BN);
                if (p.epi_bytes) {
                    // TMA-store epilogue: the warp's 32 rows leave in 32x32 chunks
                    // staged in shared memory (64-byte swizzle, two buffers)
                    if (!any) continue;
                    // one 32-column chunk: stage in the next buffer, store by TMA
                    // (with_bias: column i's bias is lane i's entry bj)
                    auto store_chunk = [&](const uint32_t (&v)[32], int j, float bj, auto with_bias) {
                        constexpr bool kBias = decltype(with_bias)::value;
                        const int n0 = t.n_tile * p.BN + 32 * j;
                        auto val = [&](int i) {
                            const float b = kBias ? __shfl_sync(0xffffffffu, bj, i) : 0.0f;
                            return __uint_as_float(v[i]) * scale + b;
                        };
                        const uint32_t buf = bufs + static_cast<uint32_t>(epi_iter & 1) * kEpiChunkBytes;
                        ++epi_iter;
                        // this buffer's last TMA store has read it (staged
                        // stores read it back synchronously)
                        if (p.epi_mode == 1 && lane == 0) bulk_wait_read<1>();
                        __syncwarp();
                        const uint32_t rowaddr = buf + static_cast<uint32_t>(lane) * 64u;
                        const uint32_t sw = static_cast<uint32_t>((lane >> 1) & 3);
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint32_t w0 = pack_bf16x2(val(8 * c + 0), val(8 * c + 1));
                            const uint32_t w1 = pack_bf16x2(val(8 * c + 2), val(8 * c + 3));
                            const uint32_t w2 = pack_bf16x2(val(8 * c + 4), val(8 * c + 5));
                            const uint32_t w3 = pack_bf16x2(val(8 * c + 6), val(8 * c + 7));
                            st_shared_v4(rowaddr + ((static_cast<uint32_t>(c) ^ sw) << 4), w0, w1, w2, w3);
                        }
                        if (p.epi_mode == 1) {
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                if (AMODE == AM_TEMPORAL)
                                    tma_store_3d(&tm.c[0], buf, n0, wrow0, plane);
                                else
                                    tma_store_2d(&tm.c[rphase], buf, n0, wrow0);
                                bulk_commit();
                            }
                            return;
                        }
                        // staged stores (rows whose byte pitch is not a
                        // multiple of 16): read the chunk back in row order
                        // and write 8-byte pieces, 4 rows of 64 bytes per
                        // instruction (K % 4 == 0), else 4-byte pieces, 2 rows
                        __syncwarp();
                        const bool wide = (p.K & 3) == 0;
                        const int rows_per = wide ? 4 : 2, lanes_per = 32 / rows_per;
                        const int piece = lane % lanes_per;             // 8- or 4-byte piece
                        for (int rr = lane / lanes_per; rr < 32; rr += rows_per) {
                            const int lr = wrow0 + rr;                  // row within the phase / plane
                            long long orow;
                            bool ok;
                            if (AMODE == AM_TEMPORAL) {
                                ok = lr < p.HW;
                                orow = static_cast<long long>(plane) * p.HW + lr;
                            } else {
                                ok = lr < phase_rows;
                                orow = static_cast<long long>(lr) * p.phases + rphase;
                            }
                            const int col = n0 + (wide ? 4 : 2) * piece;
                            if (!ok || col >= p.K) continue;
                            const int byte = (wide ? 8 : 4) * piece;     // within the 64-byte row
                            const uint32_t a = buf + static_cast<uint32_t>(rr) * 64u +
                                               ((static_cast<uint32_t>((byte >> 4) ^ ((rr >> 1) & 3)) << 4) |
                                                static_cast<uint32_t>(byte & 15));
                            __nv_bfloat16* dst = out + orow * p.K + col;
                            if (wide) {
                                *reinterpret_cast<uint2*>(dst) = ld_shared_v2(a);
                            } else {
                                uint32_t v1;
                                asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v1) : "r"(a) : "memory");
                                *reinterpret_cast<uint32_t*>(dst) = v1;
                            }
                        }
                    };
                    // chunks holding columns below K; the TMEM load of chunk
                    // j + 1 is in flight while chunk j is converted and stored
                    const int nch = min(p.BN / 32, (p.K - t.n_tile * p.BN + 31) / 32);
                    uint32_t va[32], vb[32];
                    auto chunk = [&](const uint32_t (&v)[32], int j, float bj) {
                        if (p.bias)
                            store_chunk(v, j, bj, std::integral_constant<bool, true>());
                        else
                            store_chunk(v, j, bj, std::integral_constant<bool, false>());
                    };
                    tmem_ld_32x32b_x32(tb, va);
#pragma unroll
                    for (int j = 0; j < 8; j += 2) {   // at most 8 chunks (BN <= 256)
                        if (j >= nch) break;
                        tmem_ld_wait();
                        if (j + 1 < nch) tmem_ld_32x32b_x32(tb + 32 * (j + 1), vb);
                        chunk(va, j, bl[j]);
                        if (j + 1 >= nch) break;
                        tmem_ld_wait();
                        if (j + 2 < nch) tmem_ld_32x32b_x32(tb + 32 * (j + 2), va);
                        chunk(vb, j + 1, bl[j + 1]);
                    }
                    continue;
                }
                for (int j = 0; j < p.BN / 32; ++j) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tb + 32 * j, v);
                    tmem_ld_wait();
                    const int n0 = t.n_tile * p.BN + 32 * j;
                    if (valid && n0 < p.K) {
                        const int cnt = min(32, p.K - n0);
                        if (p.splits == 1) {
                            if (p.act == kActNone)
                                store_row_bf16(out + m * p.K + n0, v, scale,
                                               p.bias ? p.bias + n0 : nullptr, cnt, vec_out);
                            else
                                store_row_bf16_act(out + m * p.K + n0, v, scale,
                                                   p.bias ? p.bias + n0 : nullptr, p.act, cnt,
                                                   vec_out);
                        } else {
                            float* dst = p.ws + (static_cast<long long>(t.split) * p.M + m) * p.K + n0;
                            store_row_f32(dst, v, cnt, vec_ws);
                        }
                    }
                }
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
        // the staging buffers are read out before the CTA leaves; the stores'
        // global writes complete with the grid (the next kernel in the
        // stream, or a dependent launch's wait, sees them)
        if (p.epi_mode == 1 && lane == 0) bulk_wait_read<0>();
    } else if (kGather) {
        // ------------------------------------------------------ row gather
        const int g = threadIdx.x - (2 + kEpiWarps) * 32;
        if (p.g_row_bytes % 8 == 0)
            gather_producer<8, 2>(p, tiles, full0, empty0, abort_flag, g);
        else
            gather_producer<4, 2>(p, tiles, full0, empty0, abort_flag, g);
    }

    __syncthreads();
    // In a pair, both CTAs finish their roles (and the peer's last remote
    // arrivals land) before either drains, frees TMEM or leaves.
    if (PAIR) cluster_sync();
    if (PAIR && *abort_flag) {
        // a pair CTA's own loads signal the leader's barriers, so it cannot
        // watch them land: after an abort both CTAs let ~100 us pass (far
        // beyond any copy's latency) before draining and leaving
        const long long t0 = clock64();
        while (clock64() - t0 < 200000) {
        }
    }
    if (*abort_flag) {
        // drain: TMA boxes armed but never waited for, then the MMAs in flight
        if (warp == 0 && lane == 0 && !kGather && rank == 0) {
            const uint32_t issued = misc[2], consumed = misc[3];
            for (uint32_t i = consumed; i < issued; ++i)
                drain_wait(full0 + 8 * (i % static_cast<uint32_t>(p.stages)),
                           (i / static_cast<uint32_t>(p.stages)) & 1u);
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

template <int AM, int F8, int PAIR>
cudaError_t launch_one(const TMaps* tm, const KParams& p, int grid, size_t smem,
                       cudaStream_t stream) {
    auto kern = conv_igemm_kernel<AM, F8, PAIR>;
    static std::atomic<int> smem_set[kMaxDevices];
    cudaError_t e = ensure_dynamic_smem(kern, smem, smem_set);
    if (e != cudaSuccess) return e;
    const int threads = (AM == AM_GEMM_GATHER) ? 320 : 192;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    // the set-up (barriers, TMEM, descriptor prefetch) may overlap the tail
    // of the previous kernel in the stream; the pdl override 0 turns this off
    if (overrides().pdl != 0) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (PAIR) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 2;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, *tm, p);
}

}  // namespace

cudaError_t launch_igemm(int amode, int fp8, const TMaps* tm, const KParams& kp, int grid,
                         size_t smem, cudaStream_t stream) {
    KParams p = kp;
    const auto u32 = [](long long v) { return static_cast<uint32_t>(v < 1 ? 1 : v); };
    p.f_tiles = make_fastdiv(u32(static_cast<long long>(p.m_tiles) * p.n_tiles));
    p.f_group = make_fastdiv(u32(static_cast<long long>(p.group_m) * p.n_tiles));
    p.f_gm = make_fastdiv(u32(p.group_m));
    p.f_planes = make_fastdiv(u32(static_cast<long long>(p.N) * p.Do));
    p.f_hw_tiles = make_fastdiv(u32(p.hw_tiles));
    p.f_Do = make_fastdiv(u32(p.Do));
    p.f_Ho = make_fastdiv(u32(p.Ho));
    p.f_Wo = make_fastdiv(u32(p.Wo));
    p.f_taps = make_fastdiv(u32(p.taps));
    p.f_S = make_fastdiv(u32(p.S));
    p.f_R = make_fastdiv(u32(p.R));
    p.rows32 = p.M + 4 * kBM < (1ll << 31) ? 1 : 0;
    const int key = (amode * 2 + (fp8 ? 1 : 0)) * 2 + (p.pair ? 1 : 0);
    switch (key) {
#define C3D_CASE(AM, F8, PR) \
    case (AM * 2 + F8) * 2 + PR: return launch_one<AM, F8, PR>(tm, p, grid, smem, stream);
        C3D_CASE(AM_IM2COL, 0, 0)
        C3D_CASE(AM_IM2COL, 1, 0)
        C3D_CASE(AM_IM2COL, 0, 1)
        C3D_CASE(AM_IM2COL, 1, 1)
        C3D_CASE(AM_TEMPORAL, 0, 0)
        C3D_CASE(AM_TEMPORAL, 1, 0)
        C3D_CASE(AM_TEMPORAL, 0, 1)
        C3D_CASE(AM_TEMPORAL, 1, 1)
        C3D_CASE(AM_GEMM_TMA, 0, 0)
        C3D_CASE(AM_GEMM_TMA, 1, 0)
        C3D_CASE(AM_GEMM_TMA, 0, 1)
        C3D_CASE(AM_GEMM_TMA, 1, 1)
        C3D_CASE(AM_GEMM_GATHER, 0, 0)
        C3D_CASE(AM_GEMM_GATHER, 1, 0)
#undef C3D_CASE
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace c3d
