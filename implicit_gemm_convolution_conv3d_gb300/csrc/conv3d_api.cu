// conv3d_api.cu -- the C ABI of libconv3d.so (declared in include/conv3d.h):
// argument checks, output dims, dispatch class, tile plan, TMA descriptor
// encoding and kernel launches.  No allocation: every buffer is the caller's.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "conv3d.h"
#include "internal.h"
#include "tile_table.h"

namespace c3d {

__device__ int g_device_status;

namespace {

thread_local char t_last_error[256] = "";

void set_error(const char* fmt, const char* a = "", long long b = 0) {
    std::snprintf(t_last_error, sizeof t_last_error, fmt, a, b);
}

int cuda_fail(cudaError_t e, const char* where) {
    std::snprintf(t_last_error, sizeof t_last_error, "%s: %s", where, cudaGetErrorString(e));
    return CONV_ERR_CUDA;
}

// ------------------------------------------------------------ driver entry points
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*EncodeIm2colFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const int*, const int*,
                                   cuuint32_t, cuuint32_t, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::once_flag g_entry_once;
EncodeTiledFn g_encode_tiled = nullptr;
EncodeIm2colFn g_encode_im2col = nullptr;

bool load_entry_points() {
    std::call_once(g_entry_once, [] {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode_tiled = reinterpret_cast<EncodeTiledFn>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode_im2col = reinterpret_cast<EncodeIm2colFn>(fn);
    });
    return g_encode_tiled != nullptr && g_encode_im2col != nullptr;
}

// ------------------------------------------------------------ per-device state
constexpr int kMaxDevices = 64;
struct DeviceInfo {
    bool ready;
    int num_sms;
    int smem_optin;
    int* status;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

int device_info(DeviceInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) {
        set_error("device ordinal out of range");
        return CONV_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_dev_mutex);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) !=
            cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (major < 10) {
            set_error("this library needs a Blackwell (sm_10x) GPU");
            return CONV_ERR_UNSUPPORTED;
        }
        if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) !=
            cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if ((e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                        dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_device_status)) != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress");
        d.status = static_cast<int*>(p);
        d.ready = true;
    }
    *out = &d;
    return CONV_OK;
}

unsigned long long g_wait_ns = 2000000000ull;

// ------------------------------------------------------------ overrides
static_assert(sizeof(Overrides) == sizeof(conv_overrides), "override layouts differ");
std::mutex g_ovr_mutex;
Overrides g_ovr = {-1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1};

// ------------------------------------------------------------ geometry
struct Geo {
    long long N, D, H, W, C, K, T, R, S;
    int sd, sh, sw, pd, ph, pw, dd, dh, dw;
    long long Do, Ho, Wo;
};

long long out_extent(long long in, long long f, int s, int p, int d) {
    const long long span = in + 2LL * p - static_cast<long long>(d) * (f - 1) - 1;
    if (span < 0) return 0;
    return span / s + 1;
}

int make_geo(const int64_t xd[5], const int64_t wd[5], const int st[3], const int pa[3],
             const int di[3], Geo* g) {
    if (!xd || !wd || !st || !pa || !di) {
        set_error("null shape argument");
        return CONV_ERR_INVALID;
    }
    for (int i = 0; i < 5; ++i)
        if (xd[i] <= 0 || wd[i] <= 0 || xd[i] > 0x7FFFFFFFll || wd[i] > 0x7FFFFFFFll) {
            set_error("dims must be in [1, 2^31)");
            return CONV_ERR_INVALID;
        }
    for (int i = 0; i < 3; ++i)
        if (st[i] <= 0 || di[i] <= 0 || pa[i] < 0) {
            set_error("strides and dilations must be positive, pads non-negative");
            return CONV_ERR_INVALID;
        }
    if (xd[4] != wd[4]) {
        set_error("x and w disagree on C");
        return CONV_ERR_INVALID;
    }
    g->N = xd[0]; g->D = xd[1]; g->H = xd[2]; g->W = xd[3]; g->C = xd[4];
    g->K = wd[0]; g->T = wd[1]; g->R = wd[2]; g->S = wd[3];
    g->sd = st[0]; g->sh = st[1]; g->sw = st[2];
    g->pd = pa[0]; g->ph = pa[1]; g->pw = pa[2];
    g->dd = di[0]; g->dh = di[1]; g->dw = di[2];
    g->Do = out_extent(g->D, g->T, g->sd, g->pd, g->dd);
    g->Ho = out_extent(g->H, g->R, g->sh, g->ph, g->dh);
    g->Wo = out_extent(g->W, g->S, g->sw, g->pw, g->dw);
    if (g->Do <= 0 || g->Ho <= 0 || g->Wo <= 0) {
        set_error("empty output");
        return CONV_ERR_INVALID;
    }
    return CONV_OK;
}

// ------------------------------------------------------------ plan
struct Plan {
    int cls, amode, fp8, elt;
    int BN, BK, stages, splits, group_m;
    long long M;
    int m_tiles, n_tiles, k_steps, taps, steps_per_split, hw_tiles, HW;
    long long g_row_bytes;   // GEMM classes: bytes of one A / B row as the caller laid it out
    long long tma_row_bytes; // GEMM classes: row pitch the TMA maps read (padded copy or caller's)
    int repack;              // 1: A and B are first copied to 16-byte aligned rows in workspace
    size_t repack_bytes;     // workspace bytes of those copies (A rows, then B rows)
    int phases;              // 2: A rows alternate 16-byte aligned / 8 bytes past (two-phase GEMM)
    int mt_phase0;           // m-tiles of phase 0 (all m-tiles when phases == 1)
    long long rows0, rows1;  // GEMM rows of phase 0 / phase 1
    size_t splitk_off;       // workspace offset of the split-K partials
    int grid;
    size_t smem;
    uint32_t tmem_cols;
    uint32_t epi_bytes;      // epilogue staging (0: direct stores from registers)
    int epi_mode;            // 0 direct, 1 TMA tensor stores, 2 staged 8- / 4-byte stores
    int pair;                // CTA-pair kernel: 256-row units on clusters of two CTAs
    int msub;                // row sub-tiles per unit sharing each B stage
    int slices;              // launches the units are cut into (whole waves each)
    int a_ncdhw;             // 1: x is channel-major (NCDHW), read as MN-major A boxes
    int ncdhw_pack;          // 1: x is channel-major, packed to an NDHWC copy in the
                             //    workspace before the conv reads it
    size_t ws_bytes;         // split-K workspace needed by this plan
};

// Bytes per k-step row: each k-step has a fixed issue cost, so the widest
// step whose padded reduction stays within 25% of the tightest padding.
int pick_bk(long long row_bytes) {
    long long tight = ((row_bytes + 31) / 32) * 32;
    for (int bk : {128, 64})
        if (((row_bytes + bk - 1) / bk) * bk * 4 <= tight * 5) return bk;
    return 32;
}

// Tile columns: a tcgen05.mma of M=128 costs about the same issue time for
// any N, so the fewest column tiles wins; among those, the narrowest tile
// (least padding in the B loads and the epilogue).
int pick_bn(long long K) {
    const long long tiles = (K + 255) / 256;
    for (int bn = 32; bn <= 256; bn += 32)
        if ((K + bn - 1) / bn == tiles) return bn;
    return 256;
}

const TileEntry* lookup_tile(int fp8, int cls, const Geo& g, long long M) {
    const long long trs = g.T * g.R * g.S;
    for (const TileEntry& e : kTileTable) {
        if (e.C == 0) continue;
        if (e.fp8 == fp8 && e.cls == cls && e.C == g.C && e.K == g.K && e.TRS == trs &&
            M >= e.m_lo && M <= e.m_hi)
            return &e;
    }
    return nullptr;
}

// Tile overrides (conv_set_overrides): a field above 0 replaces the plan's value.
void force_tile(const Overrides& o, int* bn, int* bk, int* st, int* grp, int* spl) {
    if (o.tile_n > 0) *bn = o.tile_n;
    if (o.k_bytes > 0) *bk = o.k_bytes;
    if (o.stages > 0) *st = o.stages;
    if (o.group_m > 0) *grp = o.group_m;
    if (o.splits > 0) *spl = o.splits;
}

bool gemm_amode(int amode) { return amode == AM_GEMM_TMA || amode == AM_GEMM_GATHER; }

long long gcd_ll(long long a, long long b) {
    while (b) {
        const long long t = a % b;
        a = b;
        b = t;
    }
    return a;
}

// Temporal class: T x 1 x 1 filter, unit H/W stride, no H/W padding.
bool temporal_class(const Geo& g) {
    return g.R == 1 && g.S == 1 && g.sh == 1 && g.sw == 1 && g.ph == 0 && g.pw == 0;
}

// im2col descriptor limits for a 5-D tensor: traversal stride <= 8, box
// corners in [-16, 15], tap offsets below 32.
bool im2col_fits(const Geo& g) {
    const int pads[3] = {g.pd, g.ph, g.pw};
    const int sts[3] = {g.sd, g.sh, g.sw};
    const long long ext[3] = {g.dd * (g.T - 1), g.dh * (g.R - 1), g.dw * (g.S - 1)};
    for (int i = 0; i < 3; ++i) {
        const long long up = pads[i] - ext[i];
        if (sts[i] > 8 || pads[i] > 16 || up < -16 || up > 15 || ext[i] > 31) return false;
    }
    return true;
}

// Non-overlapping patches (stride == filter, zero padding; dilation can only
// matter for a filter extent above 1) that neither implicit class can read:
// channel rows not a multiple of 16 bytes, or strides beyond the im2col box.
// Patches covering all of x are the point-output class instead.
bool patch_gather_class(const Geo& g, long long elt) {
    const bool patches = g.pd == 0 && g.ph == 0 && g.pw == 0 && g.sd == g.T && g.sh == g.R &&
                         g.sw == g.S && (g.dd == 1 || g.T == 1) && (g.dh == 1 || g.R == 1) &&
                         (g.dw == 1 || g.S == 1);
    if (!patches) return false;
    const bool implicit = (g.C * elt) % 16 == 0 && (temporal_class(g) || im2col_fits(g));
    return !implicit;
}

// ws_avail: workspace bytes the call can use (SIZE_MAX: plan the preferred
// layout and report its size).  Split-K partials and the aligned operand
// copies of the point-output GEMM are used only when they fit.
// Channel planes (D*H*W elements of one channel) up to this size are read in
// place from a channel-major x; larger ones are packed first when the filter
// has several taps.
constexpr long long kInPlaceChannelBytes = 1ll << 20;

// ncdhw: x is channel-major [N, C, D, H, W] (g keeps the NDHWC names); only
// the temporal class reads it, as MN-major A boxes of H*W positions, or from
// an NDHWC copy packed into the workspace (ncdhw_pack).
// act: the epilogue activation (plans with one store through the direct path).
int make_plan(const Geo& g, int dtype, int num_sms, int smem_optin, size_t ws_avail, Plan* P,
              bool ncdhw = false, int act = kActNone) {
    if (dtype != CONV_DTYPE_BF16 && dtype != CONV_DTYPE_FP8_E4M3) {
        set_error("unknown dtype");
        return CONV_ERR_INVALID;
    }
    std::memset(P, 0, sizeof *P);
    const Overrides ov = overrides();
    P->fp8 = dtype == CONV_DTYPE_FP8_E4M3;
    P->elt = P->fp8 ? 1 : 2;
    const long long elt = P->elt;
    if (ncdhw) {
        // a position-contiguous A tile needs the filter to leave H and W
        // alone; TMA needs 16-byte plane and filter-row pitches
        if (P->fp8) {
            set_error("channel-major x: bf16 only");
            return CONV_ERR_UNSUPPORTED;
        }
        if (!temporal_class(g)) {
            set_error("channel-major x: T x 1 x 1 filters, unit H/W stride, no H/W padding");
            return CONV_ERR_UNSUPPORTED;
        }
        if ((g.H * g.W) % 8 != 0 || (g.C * elt) % 16 != 0) {
            set_error("channel-major x: H*W and C must be multiples of 8");
            return CONV_ERR_UNSUPPORTED;
        }
        // In-place reads touch one page per channel plane per tile: with
        // channel planes past about 1 MB (a 2 MB page each) and every plane
        // read again by the other taps, the translations miss and L2 reuse
        // collapses (3x the DRAM reads, 1.8x the time on the 3x1x1 workload).
        // There, when the workspace holds an NDHWC copy, x is packed into it
        // first (6.4 ms against 8.7 ms in place on that workload).
        // The ncdhw_in_place override keeps in-place reads.
        const size_t xcopy =
            static_cast<size_t>((g.N * g.C * g.D * g.H * g.W * elt + 255) / 256 * 256);
        if (g.T > 1 && g.D * g.H * g.W * elt > kInPlaceChannelBytes && g.C % 16 == 0 &&
            ws_avail >= xcopy && ov.ncdhw_in_place != 1) {
            P->ncdhw_pack = 1;
            P->repack_bytes = xcopy;
        } else {
            P->a_ncdhw = 1;
        }
    }
    const bool zero_pad = g.pd == 0 && g.ph == 0 && g.pw == 0;
    const bool unit_stride = g.sd == 1 && g.sh == 1 && g.sw == 1;
    const bool point_output = zero_pad && g.D == g.T && g.H == g.R && g.W == g.S;
    const bool pointwise = g.T == 1 && g.R == 1 && g.S == 1 && unit_stride && zero_pad;
    long long rg = 0;   // GEMM reduction length (elements)
    if (!ncdhw && (point_output || pointwise)) {
        P->cls = CONV_CLASS_POINT_GEMM;
        P->M = point_output ? g.N : g.N * g.D * g.H * g.W;
        rg = point_output ? g.T * g.R * g.S * g.C : g.C;
        P->g_row_bytes = rg * elt;
        P->tma_row_bytes = P->g_row_bytes;
        if (P->g_row_bytes % 16 == 0) {
            P->amode = AM_GEMM_TMA;
        } else if (P->g_row_bytes % 16 == 8 && P->M >= 2 && ov.two_phase != 0 &&
                   ws_avail >= 2 * static_cast<size_t>((g.K * (P->g_row_bytes + 8) + 255) / 256 * 256)) {
            // rows of g_row_bytes = 16q + 8: even rows start 16-byte aligned, odd
            // rows 8 bytes past a boundary.  Two row phases, each a TMA-tiled
            // GEMM over the caller's x: phase 0 reads even rows in place, phase 1
            // odd rows from 8 bytes earlier (the previous row's last 8 bytes)
            // against a weight copy shifted right by 8 zero bytes, which cancels
            // them.  Only the weights are copied (twice, to 16-byte rows).
            P->amode = AM_GEMM_TMA;
            P->phases = 2;
            P->repack = 1;
            P->tma_row_bytes = P->g_row_bytes + 8;
            P->repack_bytes =
                2 * static_cast<size_t>((g.K * P->tma_row_bytes + 255) / 256 * 256);
            P->rows0 = (P->M + 1) / 2;
            P->rows1 = P->M / 2;
        } else if (P->g_row_bytes % 4 == 0) {
            // rows the TMA cannot address: copy both operands to 16-byte
            // aligned, zero-padded rows when the workspace allows it (a
            // short copy kernel, then TMA tiles), else gather with cp.async
            const long long pitch = (P->g_row_bytes + 15) / 16 * 16;
            const size_t a_bytes = static_cast<size_t>((P->M * pitch + 255) / 256 * 256);
            const size_t b_bytes = static_cast<size_t>((g.K * pitch + 255) / 256 * 256);
            if (ws_avail >= a_bytes + b_bytes && ov.repack != 0) {
                P->amode = AM_GEMM_TMA;
                P->repack = 1;
                P->repack_bytes = a_bytes + b_bytes;
                P->tma_row_bytes = pitch;
            } else {
                P->amode = AM_GEMM_GATHER;
            }
        } else {
            set_error("point-output GEMM needs T*R*S*C*elem_bytes %% 4 == 0");
            return CONV_ERR_UNSUPPORTED;
        }
    } else if (!ncdhw && patch_gather_class(g, elt)) {
        // stride == filter, output larger than one point, and the implicit
        // classes cannot read x (channel rows or strides TMA cannot address):
        // gather the non-overlapping patches into GEMM rows, then one GEMM
        P->cls = CONV_CLASS_PATCH_GEMM;
        P->M = g.N * g.Do * g.Ho * g.Wo;
        rg = g.T * g.R * g.S * g.C;
        P->g_row_bytes = rg * elt;
        P->tma_row_bytes = (P->g_row_bytes + 15) / 16 * 16;
        P->amode = AM_GEMM_TMA;
        P->repack = 2;
        P->repack_bytes = static_cast<size_t>((P->M * P->tma_row_bytes + 255) / 256 * 256);
        if (P->tma_row_bytes != P->g_row_bytes)   // weight rows copied to the pitch too
            P->repack_bytes += static_cast<size_t>((g.K * P->tma_row_bytes + 255) / 256 * 256);
        if (ws_avail < P->repack_bytes) {
            set_error("the patch gather needs %s%lld bytes of workspace (conv_fwd_plan)", "",
                      static_cast<long long>(P->repack_bytes));
            return CONV_ERR_INVALID;
        }
    } else {
        if ((g.C * elt) % 16 != 0) {
            set_error("implicit GEMM needs C*elem_bytes %% 16 == 0");
            return CONV_ERR_UNSUPPORTED;
        }
        P->M = g.N * g.Do * g.Ho * g.Wo;
        if (g.R == 1 && g.S == 1 && g.sh == 1 && g.sw == 1 && g.ph == 0 && g.pw == 0) {
            P->cls = CONV_CLASS_TEMPORAL;
            P->amode = AM_TEMPORAL;
            if (g.H * g.W > 0x7FFFFFFFll || g.D > 0x7FFFFFFFll) {
                set_error("temporal plane too large");
                return CONV_ERR_UNSUPPORTED;
            }
        } else {
            P->cls = CONV_CLASS_GENERIC;
            P->amode = AM_IM2COL;
            // im2col descriptor limits for a 5-D tensor: traversal stride <= 8, box
            // corners in [-16, 15], tap offsets below 32
            const int pads[3] = {g.pd, g.ph, g.pw};
            const int sts[3] = {g.sd, g.sh, g.sw};
            const long long ext[3] = {g.dd * (g.T - 1), g.dh * (g.R - 1), g.dw * (g.S - 1)};
            for (int i = 0; i < 3; ++i) {
                const long long up = pads[i] - ext[i];
                if (sts[i] > 8 || pads[i] > 16 || up < -16 || up > 15 || ext[i] > 31) {
                    set_error("im2col limits: stride <= 8, pad <= 16, dilated filter extent <= 32");
                    return CONV_ERR_UNSUPPORTED;
                }
            }
        }
    }
    if (P->M > 0x7FFFFFFFll * 128ll) {
        set_error("too many output rows");
        return CONV_ERR_UNSUPPORTED;
    }

    // tile defaults
    int BN = pick_bn(g.K);
    int BK = (P->amode == AM_GEMM_GATHER)
                 ? 128
                 : pick_bk(gemm_amode(P->amode) ? P->tma_row_bytes : g.C * elt);
    // raster group 1: a unit's row block meets every column tile before the
    // next row block starts (best on the measured workloads)
    int stages = 0, group_m = 1, splits = 0, pair_pref = -1, msub_pref = 0;
    if (const TileEntry* e = lookup_tile(P->fp8, P->cls, g, P->M)) {
        if (e->BN) BN = e->BN;
        if (e->BK) BK = e->BK;
        if (e->stages) stages = e->stages;
        if (e->group_m) group_m = e->group_m;
        if (e->splits) splits = e->splits;
        pair_pref = e->pair;
        msub_pref = e->msub;
    }
    force_tile(ov, &BN, &BK, &stages, &group_m, &splits);
    // MN-major A boxes are 64 channel rows of 128 bytes: 128- or 256-byte k-steps
    if (P->a_ncdhw && BK < 128) BK = 128;
    if (BN < 32 || BN > 256 || BN % 32 != 0 || !(BK == 32 || BK == 64 || BK == 128 || BK == 256) ||
        (P->amode == AM_GEMM_GATHER && BK != 128) || group_m < 1) {
        set_error("invalid tile override");
        return CONV_ERR_INVALID;
    }
    P->BN = BN;
    P->BK = BK;
    P->group_m = group_m;

    if (gemm_amode(P->amode)) {
        P->taps = 1;
        P->k_steps = static_cast<int>((P->tma_row_bytes + BK - 1) / BK);
    } else {
        P->taps = static_cast<int>(g.T * g.R * g.S);
        const long long chunks = (g.C * elt + BK - 1) / BK;
        P->k_steps = static_cast<int>(chunks * P->taps);
    }
    if (P->phases != 2) {
        P->phases = 1;
        P->rows0 = P->M;
        P->rows1 = 0;
    }
    auto set_m_tiles = [&](int tile_m) {
        if (P->cls == CONV_CLASS_TEMPORAL) {
            P->HW = static_cast<int>(g.H * g.W);
            P->hw_tiles = (P->HW + tile_m - 1) / tile_m;
            P->m_tiles = static_cast<int>(g.N * g.Do * P->hw_tiles);
            P->mt_phase0 = P->m_tiles;
        } else if (P->phases == 2) {
            P->mt_phase0 = static_cast<int>((P->rows0 + tile_m - 1) / tile_m);
            P->m_tiles = P->mt_phase0 + static_cast<int>((P->rows1 + tile_m - 1) / tile_m);
        } else {
            P->m_tiles = static_cast<int>((P->M + tile_m - 1) / tile_m);
            P->mt_phase0 = P->m_tiles;
        }
    };
    set_m_tiles(kBM);
    P->n_tiles = static_cast<int>((g.K + BN - 1) / BN);

    // split-K when the output tiles leave most SMs idle
    const long long tiles = static_cast<long long>(P->m_tiles) * P->n_tiles;
    if (splits == 0) {
        splits = 1;
        if (tiles * 2 <= num_sms && P->k_steps >= 4)
            splits = static_cast<int>(std::min<long long>({num_sms / tiles, P->k_steps / 2, 32}));
    }
    splits = std::max(1, std::min(splits, P->k_steps));
    P->steps_per_split = (P->k_steps + splits - 1) / splits;
    splits = (P->k_steps + P->steps_per_split - 1) / P->steps_per_split;
    const size_t splitk_bytes =
        splits > 1 ? static_cast<size_t>(splits) * P->M * g.K * sizeof(float) : 0;
    P->splitk_off = P->repack_bytes;
    if (splits > 1 && ws_avail < P->repack_bytes + splitk_bytes) {
        splits = 1;
        P->steps_per_split = P->k_steps;
    }
    P->ws_bytes = P->repack_bytes + (splits > 1 ? splitk_bytes : 0);
    P->splits = splits;
    if (tiles * splits > 0x7FFFFFFFll) {
        set_error("too many work units");
        return CONV_ERR_UNSUPPORTED;
    }

    // CTA pairs (tcgen05 cta_group::2): a cluster of two CTAs computes a
    // 256-row unit, each SM holding half of the B tile, which halves the B
    // bytes each SM stores and feeds to the tensor core.  Used when the
    // problem has whole waves of such units; the pair override decides otherwise.
    P->pair = 0;
    if (P->amode != AM_GEMM_GATHER && splits == 1 && BN >= 64 && num_sms % 2 == 0) {
        const long long pm = P->cls == CONV_CLASS_TEMPORAL
                                 ? g.N * g.Do * ((g.H * g.W + 2 * kBM - 1) / (2 * kBM))
                                 : (P->M + 2 * kBM - 1) / (2 * kBM);
        int want = pm * P->n_tiles >= 2LL * num_sms ? 1 : 0;
        if (pair_pref >= 0) want = pair_pref;
        if (ov.pair >= 0) want = ov.pair ? 1 : 0;
        if (want) {
            P->pair = 1;
            set_m_tiles(2 * kBM);
        }
    }
    // Two row sub-tiles per unit share every B stage (two accumulators in
    // TMEM, no epilogue overlap): halves the B bytes per flop, for long
    // reductions where the exposed epilogue is a small share of the unit.
    P->msub = 1;
    if (P->amode != AM_GEMM_GATHER && splits == 1 && 2 * BN <= 256 + 256) {
        const int rows = (2 * kBM) << P->pair;
        const long long mt = P->cls == CONV_CLASS_TEMPORAL
                                 ? g.N * g.Do * ((g.H * g.W + rows - 1) / rows)
                                 : (P->M + rows - 1) / rows;
        int want = (P->k_steps >= 384 && mt * P->n_tiles >= 2LL * (num_sms >> P->pair)) ? 2 : 1;
        if (msub_pref > 0) want = msub_pref;
        if (ov.msub > 0) want = ov.msub == 2 ? 2 : 1;
        if (want == 2) {
            P->msub = 2;
            set_m_tiles(rows);
        }
    }

    // bf16 output leaves through TMA stores when its rows are 16-byte aligned
    // (a warp's 32 rows x 64 bytes per store, where direct stores would send
    // 32 separate 16-byte pieces per instruction); split-K partials are
    // written directly
    // bf16 rows of an even K whose pitch is not a multiple of 16 bytes are
    // staged the same way and leave in 8- or 4-byte pieces, several rows per
    // instruction, instead of 2-byte stores from each lane's own row
    // An activation is applied on the direct-store path only, which keeps one
    // compiled copy of its code out of the staged epilogues (their code size
    // is what the short point-output kernels are sensitive to).
    P->epi_mode = splits > 1 || act != kActNone ? 0 : (g.K % 8 == 0 ? 1 : (g.K % 2 == 0 ? 2 : 0));
    // the epilogue override (1 TMA, 2 staged, 3 direct) where the shape allows it
    if (act == kActNone) {
        if (ov.epilogue == 1 && splits == 1 && g.K % 8 == 0) P->epi_mode = 1;
        if (ov.epilogue == 2 && splits == 1 && g.K % 2 == 0) P->epi_mode = 2;
        if (ov.epilogue == 3) P->epi_mode = 0;
    }
    P->epi_bytes = P->epi_mode ? kEpiStageBytes : 0u;
    // pipeline depth from the shared-memory budget (a pair CTA holds half of B)
    const size_t stage_bytes = static_cast<size_t>(P->msub * kBM + (BN >> P->pair)) * BK;
    const size_t fixed = 1024 + 256 + P->epi_bytes;
    const int max_stages = static_cast<int>((smem_optin - fixed) / stage_bytes);
    if (stages == 0) stages = std::min(8, max_stages);
    const int min_stages = (P->amode == AM_GEMM_GATHER) ? 3 : 2;
    if (stages < min_stages || stages > max_stages) {
        set_error("pipeline depth out of range for this tile");
        return CONV_ERR_UNSUPPORTED;
    }
    P->stages = stages;
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(2 * BN)) cols <<= 1;
    P->tmem_cols = cols;
    P->smem = fixed + stage_bytes * stages;
    // a CTA holding all 512 TMEM columns must be alone on its SM
    if (cols > 256 && P->smem < static_cast<size_t>(smem_optin) / 2 + 1024)
        P->smem = static_cast<size_t>(smem_optin) / 2 + 1024;
    const long long units = static_cast<long long>(P->m_tiles) * P->n_tiles * splits;
    if (P->pair)
        P->grid = 2 * static_cast<int>(std::min<long long>(units, num_sms / 2));
    else
        P->grid = static_cast<int>(std::min<long long>(units, num_sms));
    // Long reductions run as several launches of whole waves: each launch
    // starts its CTAs together, so units sharing weight slices stay in step
    // and find them in L2 (one persistent launch drifts apart over ~44 waves:
    // 27 GB of DRAM traffic per launch against 13 GB sliced on the 3x3x3
    // video conv, 1.6-4.5% faster under the power cap).  The slices override
    // sets the count (1: one launch).
    P->slices = 1;
    if (!gemm_amode(P->amode) && splits == 1) {
        const long long wave = P->grid >> P->pair;
        const long long nb = P->m_tiles / (wave / gcd_ll(wave, P->n_tiles));
        if (P->k_steps >= 384 && nb >= 4) P->slices = static_cast<int>(std::min<long long>(nb, 32));
        if (ov.slices > 0) P->slices = std::min(32, ov.slices);
    }
    return CONV_OK;
}

// ------------------------------------------------------------ tensor maps
// A 256-byte k-step is two 128-byte boxes per operand, each in the 128-byte
// swizzle; narrower k-steps are one box whose row width sets the swizzle.
CUtensorMapSwizzle swizzle_for(int bk) {
    return bk >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                     : (bk == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}

uint32_t desc_layout_for(int bk) { return bk >= 128 ? 2u : (bk == 64 ? 4u : 6u); }

int box_bytes(int bk) { return bk < 128 ? bk : 128; }

int encode_tiled(CUtensorMap* m, int fp8, int rank, const void* ptr, const cuuint64_t* dims,
                 const cuuint64_t* strides, const cuuint32_t* box, int bk) {
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode_tiled(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                rank, const_cast<void*>(ptr), dims, strides, box, es,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(bk),
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (code %s%lld)", "", static_cast<long long>(r));
        return CONV_ERR_CUDA;
    }
    return CONV_OK;
}

// The NCDHW -> NDHWC pack of x [N, C, S] (S = D*H*W): by the TMA-fed kernel
// when C and S are multiples of 8 (the box rows need 16-byte pitches) and
// its ring fits, else by the register-blocked / generic kernels (also when
// the pack_lanes override asks for the register-blocked warp tile).
cudaError_t pack_launch(const void* in, long long N, long long C, long long S, void* out, int fp8,
                        const unsigned int* amax_bits, float* scale_out, const DeviceInfo* dev,
                        cudaStream_t stream) {
    const int lanes = overrides().pack_lanes;
    if (C % 8 == 0 && S % 8 == 0 && lanes != 2 && lanes != 4 &&
        pack_tma_stages(fp8, dev->smem_optin) >= 2 && load_entry_points() && N <= 0x7FFFFFFFll) {
        CUtensorMap m;
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(C),
                                    static_cast<cuuint64_t>(N)};
        const cuuint64_t str[2] = {static_cast<cuuint64_t>(S) * 2, static_cast<cuuint64_t>(C * S) * 2};
        const cuuint32_t box[3] = {256, 128, 1};
        const cuuint32_t es[3] = {1, 1, 1};
        if (g_encode_tiled(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(in), dims,
                           str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
            return launch_pack_tma(&m, N, C, S, out, fp8, amax_bits, scale_out, dev->num_sms,
                                   dev->smem_optin, dev->status, g_wait_ns, stream);
    }
    return launch_pack(in, N, C, S, out, fp8, amax_bits, scale_out, dev->num_sms, stream);
}

// Output map for the TMA-store epilogue: [M, K] bf16 rows (or, for the
// temporal class, [N*Do planes, H*W, K] so stores clip at each plane's edge),
// 32x32 boxes with the 64-byte swizzle the epilogue writes.
int build_out_map(const Geo& g, const Plan& P, void* out, TMaps* tm) {
    std::memset(tm->c, 0, sizeof tm->c);
    if (P.epi_mode != 1) return CONV_OK;
    const cuuint64_t row = static_cast<cuuint64_t>(g.K) * 2;
    if (P.amode == AM_TEMPORAL) {
        const cuuint64_t hw = static_cast<cuuint64_t>(P.HW);
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(g.K), hw,
                                    static_cast<cuuint64_t>(g.N * g.Do)};
        const cuuint64_t str[2] = {row, row * hw};
        const cuuint32_t box[3] = {32, 32, 1};
        return encode_tiled(&tm->c[0], 0, 3, out, dims, str, box, 64);
    }
    // phase j's output rows are rows j, j + phases, ... of out
    for (int j = 0; j < P.phases; ++j) {
        const cuuint64_t rows = static_cast<cuuint64_t>(j ? P.rows1 : P.rows0);
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(g.K), rows};
        const cuuint64_t str[1] = {row * static_cast<cuuint64_t>(P.phases)};
        const cuuint32_t box[2] = {32, 32};
        int rc = encode_tiled(&tm->c[j], 0, 2, static_cast<unsigned char*>(out) + j * row, dims,
                              str, box, 64);
        if (rc) return rc;
    }
    return CONV_OK;
}

int build_maps(const Geo& g, const Plan& P, const void* x, const void* w, TMaps* tm) {
    CUtensorMap* tmA = &tm->a[0];
    CUtensorMap* tmB = &tm->b[0];
    std::memset(tm->a, 0, sizeof tm->a);
    std::memset(tm->b, 0, sizeof tm->b);
    const cuuint64_t elt = static_cast<cuuint64_t>(P.elt);
    // elements of one box row (a 256-byte k-step loads two boxes)
    const cuuint32_t bke = static_cast<cuuint32_t>(box_bytes(P.BK) / P.elt);
    if (P.amode == AM_GEMM_GATHER) return CONV_OK;
    if (P.amode == AM_GEMM_TMA && P.phases == 2) {
        // x as given: phase j's rows start j*(row - 8) bytes into x, 2*row
        // bytes apart, (row + 8*j) bytes long; w: the two aligned copies
        // (plain, and shifted right by 8 zero bytes) in the workspace
        const cuuint64_t rb = static_cast<cuuint64_t>(P.g_row_bytes);
        const cuuint64_t pitch = static_cast<cuuint64_t>(P.tma_row_bytes);
        const unsigned char* xb = static_cast<const unsigned char*>(x);
        const unsigned char* wb = static_cast<const unsigned char*>(w);
        const size_t wcopy = static_cast<size_t>((g.K * P.tma_row_bytes + 255) / 256 * 256);
        for (int j = 0; j < 2; ++j) {
            const cuuint64_t adims[2] = {(rb + 8 * j) / elt,
                                         static_cast<cuuint64_t>(j ? P.rows1 : P.rows0)};
            const cuuint64_t astr[1] = {2 * rb};
            const cuuint32_t abox[2] = {bke, static_cast<cuuint32_t>(kBM)};
            int rc = encode_tiled(&tm->a[j], P.fp8, 2, xb + j * (rb - 8), adims, astr, abox, P.BK);
            if (rc) return rc;
            const cuuint64_t bdims[2] = {pitch / elt, static_cast<cuuint64_t>(g.K)};
            const cuuint64_t bstr[1] = {pitch};
            const cuuint32_t bbox[2] = {bke, static_cast<cuuint32_t>(P.BN >> P.pair)};
            rc = encode_tiled(&tm->b[j], P.fp8, 2, wb + j * wcopy, bdims, bstr, bbox, P.BK);
            if (rc) return rc;
        }
        return CONV_OK;
    }
    if (P.amode == AM_GEMM_TMA) {
        const cuuint64_t rg = static_cast<cuuint64_t>(P.tma_row_bytes) / elt;
        const cuuint64_t adims[2] = {rg, static_cast<cuuint64_t>(P.M)};
        const cuuint64_t astr[1] = {static_cast<cuuint64_t>(P.tma_row_bytes)};
        const cuuint32_t abox[2] = {bke, static_cast<cuuint32_t>(kBM)};
        int rc = encode_tiled(tmA, P.fp8, 2, x, adims, astr, abox, P.BK);
        if (rc) return rc;
        const cuuint64_t bdims[2] = {rg, static_cast<cuuint64_t>(g.K)};
        const cuuint32_t bbox[2] = {bke, static_cast<cuuint32_t>(P.BN >> P.pair)};
        return encode_tiled(tmB, P.fp8, 2, w, bdims, astr, bbox, P.BK);
    }
    // weight: [K, T*R*S, C] -> dims {C, TRS, K}, box {bke, 1, BN}
    {
        const cuuint64_t trs = static_cast<cuuint64_t>(g.T * g.R * g.S);
        const cuuint64_t bdims[3] = {static_cast<cuuint64_t>(g.C), trs, static_cast<cuuint64_t>(g.K)};
        const cuuint64_t bstr[2] = {static_cast<cuuint64_t>(g.C) * elt,
                                    static_cast<cuuint64_t>(g.C) * elt * trs};
        const cuuint32_t bbox[3] = {bke, 1, static_cast<cuuint32_t>(P.BN >> P.pair)};
        int rc = encode_tiled(tmB, P.fp8, 3, w, bdims, bstr, bbox, P.BK);
        if (rc) return rc;
    }
    const cuuint64_t row = static_cast<cuuint64_t>(g.C) * elt;
    if (P.amode == AM_TEMPORAL && P.a_ncdhw) {
        // x as [N, C, D, H*W] -> dims {HW, D, C, N}, box {64, 1, 64, 1}:
        // 64 channel rows of 64 positions, the MN-major 128-byte swizzle atom
        const cuuint64_t hw = static_cast<cuuint64_t>(g.H * g.W);
        const cuuint64_t plane = hw * elt;
        const cuuint64_t adims[4] = {hw, static_cast<cuuint64_t>(g.D), static_cast<cuuint64_t>(g.C),
                                     static_cast<cuuint64_t>(g.N)};
        const cuuint64_t astr[3] = {plane, plane * static_cast<cuuint64_t>(g.D),
                                    plane * static_cast<cuuint64_t>(g.D * g.C)};
        const cuuint32_t abox[4] = {64, 1, bke, 1};
        return encode_tiled(tmA, 0, 4, x, adims, astr, abox, 128);
    }
    if (P.amode == AM_TEMPORAL) {
        // x as [N, D, H*W, C] -> dims {C, HW, D, N}, box {bke, 128, 1, 1}
        const cuuint64_t hw = static_cast<cuuint64_t>(g.H * g.W);
        const cuuint64_t adims[4] = {static_cast<cuuint64_t>(g.C), hw, static_cast<cuuint64_t>(g.D),
                                     static_cast<cuuint64_t>(g.N)};
        const cuuint64_t astr[3] = {row, row * hw, row * hw * static_cast<cuuint64_t>(g.D)};
        const cuuint32_t abox[4] = {bke, static_cast<cuuint32_t>(kBM), 1, 1};
        return encode_tiled(tmA, P.fp8, 4, x, adims, astr, abox, P.BK);
    }
    // generic: im2col over NDHWC -> dims {C, W, H, D, N}
    const cuuint64_t adims[5] = {static_cast<cuuint64_t>(g.C), static_cast<cuuint64_t>(g.W),
                                 static_cast<cuuint64_t>(g.H), static_cast<cuuint64_t>(g.D),
                                 static_cast<cuuint64_t>(g.N)};
    const cuuint64_t astr[4] = {row, row * static_cast<cuuint64_t>(g.W),
                                row * static_cast<cuuint64_t>(g.W * g.H),
                                row * static_cast<cuuint64_t>(g.W * g.H * g.D)};
    // bounding box of window corners along {W, H, D}: [-pad, extent - 1 + pad - dil*(f-1)]
    const int lower[3] = {-g.pw, -g.ph, -g.pd};
    const int upper[3] = {g.pw - g.dw * static_cast<int>(g.S - 1), g.ph - g.dh * static_cast<int>(g.R - 1),
                          g.pd - g.dd * static_cast<int>(g.T - 1)};
    const cuuint32_t es[5] = {1, static_cast<cuuint32_t>(g.sw), static_cast<cuuint32_t>(g.sh),
                              static_cast<cuuint32_t>(g.sd), 1};
    CUresult r = g_encode_im2col(
        tmA, P.fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5,
        const_cast<void*>(x), adims, astr, lower, upper, bke, static_cast<cuuint32_t>(kBM), es,
        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(P.BK), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeIm2col failed (code %s%lld)", "", static_cast<long long>(r));
        return CONV_ERR_CUDA;
    }
    return CONV_OK;
}

uint32_t make_idesc(int fp8, int bn, int m) {
    uint32_t d = 0;
    d |= 1u << 4;                       // D format: f32
    if (!fp8) d |= (1u << 7) | (1u << 10);   // A, B format: bf16 (kind::f16); e4m3 = 0 (kind::f8f6f4)
    d |= static_cast<uint32_t>(bn >> 3) << 17;   // N >> 3
    d |= static_cast<uint32_t>(m >> 4) << 24;    // M >> 4
    return d;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Kernel parameters of plan P over the whole problem (m-tiles [0, m_tiles)).
void fill_params(const Geo& g, const Plan& P, const void* x, const void* w, void* out,
                 void* workspace, const float* scale_x, const float* scale_w, const float* bias,
                 int* status, KParams* kp) {
    KParams& k = *kp;
    std::memset(&k, 0, sizeof k);
    k.N = static_cast<int>(g.N); k.D = static_cast<int>(g.D); k.H = static_cast<int>(g.H);
    k.W = static_cast<int>(g.W); k.C = static_cast<int>(g.C);
    k.T = static_cast<int>(g.T); k.R = static_cast<int>(g.R); k.S = static_cast<int>(g.S);
    k.Do = static_cast<int>(g.Do); k.Ho = static_cast<int>(g.Ho); k.Wo = static_cast<int>(g.Wo);
    k.sd = g.sd; k.sh = g.sh; k.sw = g.sw; k.pd = g.pd; k.ph = g.ph; k.pw = g.pw;
    k.dd = g.dd; k.dh = g.dh; k.dw = g.dw;
    k.M = P.M;
    k.K = static_cast<int>(g.K);
    k.HW = P.HW;
    k.hw_tiles = P.hw_tiles;
    // temporal units of one wave share input planes in L2 when H*W-tile
    // major; the hw_major override 0 keeps output row order
    k.hw_major = (P.cls == CONV_CLASS_TEMPORAL && overrides().hw_major != 0) ? 1 : 0;
    k.m_tiles = P.m_tiles;
    k.n_tiles = P.n_tiles;
    k.splits = P.splits;
    k.m_tile0 = 0;
    k.phases = P.phases;
    k.mt_phase0 = P.mt_phase0;
    k.rows0 = P.rows0;
    k.rows1 = P.rows1;
    k.k_steps = P.k_steps;
    k.steps_per_split = P.steps_per_split;
    k.taps = P.taps;
    k.group_m = P.group_m;
    k.BN = P.BN;
    k.BK = P.BK;
    k.stages = P.stages;
    k.a_stage_bytes = static_cast<uint32_t>(P.msub * kBM * P.BK);
    k.b_stage_bytes = static_cast<uint32_t>((P.BN >> P.pair) * P.BK);
    k.stage_bytes = k.a_stage_bytes + k.b_stage_bytes;
    k.idesc = make_idesc(P.fp8, P.BN, kBM << P.pair);
    k.layout = desc_layout_for(P.BK);
    k.sbo = static_cast<uint32_t>(8 * box_bytes(P.BK));
    k.tmem_cols = P.tmem_cols;
    k.epi_bytes = P.epi_bytes;
    k.epi_mode = P.epi_mode;
    k.pair = P.pair;
    k.msub = P.msub;
    k.ga = static_cast<const unsigned char*>(x);
    k.gb = static_cast<const unsigned char*>(w);
    k.g_row_bytes = P.g_row_bytes;
    k.out = out;
    k.ws = P.splits > 1
               ? reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + P.splitk_off)
               : nullptr;
    k.scale_x = scale_x;
    k.scale_w = scale_w;
    k.bias = bias;
    k.status = status;
    k.wait_ns = g_wait_ns;
    if (P.a_ncdhw) {
        k.a_mn = 1;
        k.idesc |= 1u << 15;   // A major-ness: MN
    }
}

// ------------------------------------------------------------ MN-major A GEMM
// out[m, n] = sum_k A[k, m] * B[n, k] (bf16 in, fp32 accumulation, bf16 out
// [M, Nn]) with A stored MN-major -- Kr rows of M contiguous elements (the
// GEMM reads it in place: TMA boxes of 64 M x 64 k and tcgen05 MN-major
// descriptors) -- and B K-major, Nn rows of Kp elements (Kp a multiple of 8,
// zero past Kr).  The backward-weights GEMM (dy is [N, K]: MN-major as the
// A of dW = dy^T x).  Plans as the pointwise GEMM of [M, Kp] by [Nn, Kp];
// returns CONV_ERR_UNSUPPORTED when that plan does not use 128-byte k-steps
// and one row sub-tile.
int gemm_mn_a(const void* a, long long M, long long Kr, const void* b, long long Nn,
              long long Kp, void* out, void* workspace, size_t workspace_bytes, DeviceInfo* dev,
              cudaStream_t stream) {
    const int64_t xi[5] = {M, 1, 1, 1, Kp}, wi[5] = {Nn, 1, 1, 1, Kp};
    const int one[3] = {1, 1, 1}, zero[3] = {0, 0, 0};
    Geo g;
    int rc = make_geo(xi, wi, one, zero, one, &g);
    if (rc) return rc;
    if (!load_entry_points()) {
        set_error("cuTensorMapEncode* entry points unavailable");
        return CONV_ERR_CUDA;
    }
    Plan P;
    if ((rc = make_plan(g, CONV_DTYPE_BF16, dev->num_sms, dev->smem_optin, workspace_bytes, &P)))
        return rc;
    if (P.amode != AM_GEMM_TMA || P.BK != 128 || P.msub != 1 || P.phases != 1 || P.repack ||
        (M * 2) % 16 != 0) {
        set_error("MN-major GEMM plan unavailable for this shape");
        return CONV_ERR_UNSUPPORTED;
    }
    TMaps tm;
    if ((rc = build_maps(g, P, a, b, &tm))) return rc;   // B (K-major) as planned
    {
        // A in place: dims {M (inner), Kr}, boxes of 64 x 64, 128-byte swizzle
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(Kr)};
        const cuuint64_t str[1] = {static_cast<cuuint64_t>(M) * 2};
        const cuuint32_t box[2] = {64, 64};
        if ((rc = encode_tiled(&tm.a[0], 0, 2, a, dims, str, box, 128))) return rc;
    }
    if ((rc = build_out_map(g, P, out, &tm))) return rc;
    KParams k;
    fill_params(g, P, a, b, out, workspace, nullptr, nullptr, nullptr, dev->status, &k);
    k.a_mn = 1;
    k.idesc |= 1u << 15;   // A major-ness: MN
    cudaError_t e = launch_igemm(P.amode, 0, &tm, k, P.grid, P.smem, stream);
    if (e != cudaSuccess) return cuda_fail(e, "conv kernel launch");
    if (P.splits > 1) {
        e = launch_splitk_reduce(k.ws, out, M * Nn, P.splits, nullptr, nullptr, nullptr, Nn, 0,
                                 dev->num_sms, stream);
        if (e != cudaSuccess) return cuda_fail(e, "split-K reduce launch");
    }
    return CONV_OK;
}

// ------------------------------------------------------------ backward passes
// Point-output geometry (MIOpen PR #10912): zero padding and the input
// spatially equal to the filter, so each batch element has one output
// position (a valid geometry with D == T forces unit dilation or T == 1).
bool is_point_output(const Geo& g) {
    return g.pd == 0 && g.ph == 0 && g.pw == 0 && g.D == g.T && g.H == g.R && g.W == g.S;
}

size_t round256(long long b) { return static_cast<size_t>((b + 255) / 256 * 256); }

// Checks shared by the two backward entry points; fills the GEMM extents
// N (batch), K (filters) and J = T*R*S*C.
int bwd_setup(const int64_t x_dims[5], const int64_t w_dims[5], const int stride[3],
              const int pad[3], const int dil[3], const void* a, const void* b, void* out,
              void* workspace, long long* N, long long* K, long long* J) {
    Geo g;
    int rc = make_geo(x_dims, w_dims, stride, pad, dil, &g);
    if (rc) return rc;
    if (!a || !b || !out) {
        set_error("null tensor pointer");
        return CONV_ERR_INVALID;
    }
    if (!aligned16(a) || !aligned16(b) || !aligned16(out) || (workspace && !aligned16(workspace))) {
        set_error("device pointers must be 16-byte aligned");
        return CONV_ERR_INVALID;
    }
    if (!is_point_output(g)) {
        set_error("backward passes cover point-output shapes only (input spatially equal to "
                  "the filter, zero padding)");
        return CONV_ERR_UNSUPPORTED;
    }
    *N = g.N;
    *K = g.K;
    *J = g.T * g.R * g.S * g.C;
    return CONV_OK;
}

// ------------------------------------------------------------ host-operand pipeline
// Per device: a copy-in and a copy-out stream and the events that order them
// against the caller's stream.  Created on first use, kept until exit.
constexpr int kMaxChunks = 32;
constexpr int kMaxWGroups = 8;   // weight copies the first slice is split over
struct Pipe {
    bool ready;
    cudaStream_t s_in, s_out;
    cudaEvent_t start, in_done, out_done;
    cudaEvent_t ev_in[kMaxChunks], ev_conv[kMaxChunks], ev_w[kMaxWGroups];
    std::mutex mu;   // one enqueue at a time per device
};
Pipe g_pipe[kMaxDevices];
std::mutex g_pipe_mutex;

int pipe_for_device(Pipe** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) {
        set_error("device ordinal out of range");
        return CONV_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_pipe_mutex);
    Pipe& p = g_pipe[dev];
    if (!p.ready) {
        if ((e = cudaStreamCreateWithFlags(&p.s_in, cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_fail(e, "cudaStreamCreateWithFlags");
        if ((e = cudaStreamCreateWithFlags(&p.s_out, cudaStreamNonBlocking)) != cudaSuccess) {
            cudaStreamDestroy(p.s_in);
            return cuda_fail(e, "cudaStreamCreateWithFlags");
        }
        cudaEvent_t* evs[3 + 2 * kMaxChunks + kMaxWGroups];
        int n = 0;
        evs[n++] = &p.start;
        evs[n++] = &p.in_done;
        evs[n++] = &p.out_done;
        for (int i = 0; i < kMaxChunks; ++i) {
            evs[n++] = &p.ev_in[i];
            evs[n++] = &p.ev_conv[i];
        }
        for (int i = 0; i < kMaxWGroups; ++i) evs[n++] = &p.ev_w[i];
        for (int i = 0; i < n; ++i) {
            if ((e = cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming)) != cudaSuccess) {
                for (int j = 0; j < i; ++j) cudaEventDestroy(*evs[j]);
                cudaStreamDestroy(p.s_in);
                cudaStreamDestroy(p.s_out);
                return cuda_fail(e, "cudaEventCreateWithFlags");
            }
        }
        p.ready = true;
    }
    *out = &p;
    return CONV_OK;
}

// Output rows [first, last) computed by m-tile mt of plan P.
long long tile_row_lo(const Plan& P, int mt) {
    const long long unit_rows = static_cast<long long>(kBM << P.pair) * P.msub;
    if (P.cls == CONV_CLASS_TEMPORAL) {
        const long long plane = mt / P.hw_tiles, hwb = mt % P.hw_tiles;
        return plane * P.HW + hwb * unit_rows;
    }
    return mt * unit_rows;
}

long long tile_row_hi(const Plan& P, int mt) {
    const long long unit_rows = static_cast<long long>(kBM << P.pair) * P.msub;
    if (P.cls == CONV_CLASS_TEMPORAL) {
        const long long plane = mt / P.hw_tiles, hwb = mt % P.hw_tiles;
        return plane * P.HW + std::min<long long>(P.HW, (hwb + 1) * unit_rows);
    }
    return std::min<long long>(P.M, (mt + 1) * unit_rows);
}

// The input that output rows [0, row_hi) read, in input planes ((n, d)
// order, H rows of W*C elements each): planes [0, whole) entirely and rows
// [0, rows) of planes [whole, part).  Output rows are output planes (n, od)
// in order, then rows oh: the output planes before the last one read, at
// most, every plane of the images before n and image n's planes up to depth
// (od-1)*sd - pd + (T-1)*dd; the last one's rows up to oh read its planes up
// to depth od*sd - pd + (T-1)*dd, input rows up to oh*sh - ph + (R-1)*dh.
struct XReach {
    long long whole, part, rows;
};

XReach x_reach(const Geo& g, long long row_hi) {
    const long long r = row_hi - 1;
    const long long oh = (r / g.Wo) % g.Ho;
    const long long q = r / (g.Wo * g.Ho);
    const long long n = q / g.Do, od = q % g.Do;
    const long long d_prev = std::min(g.D - 1, (od - 1) * g.sd - g.pd + (g.T - 1) * g.dd);
    const long long d_last = std::min(g.D - 1, od * g.sd - g.pd + (g.T - 1) * g.dd);
    const long long h = std::min(g.H - 1, oh * g.sh - g.ph + (g.R - 1) * g.dh);
    XReach x;
    x.whole = n * g.D + (od >= 1 ? std::max(d_prev, -1LL) + 1 : 0);
    x.part = std::max(x.whole, n * g.D + std::max(d_last, -1LL) + 1);
    x.rows = h < 0 ? 0 : h + 1;
    return x;
}

// Copy (host to device, on stream s) the input rows within `need` that
// `have` does not hold; ranges that meet go as one copy.
cudaError_t copy_x_reach(const Geo& g, const XReach& have, const XReach& need,
                         size_t plane_bytes, size_t row_bytes, const unsigned char* xh,
                         unsigned char* xd, cudaStream_t s) {
    auto held = [&](const XReach& r, long long p) {
        return p < r.whole ? g.H : (p < r.part ? r.rows : 0);
    };
    size_t lo = 0, hi = 0;
    for (long long p = have.whole; p < need.part; ++p) {
        const long long a = held(have, p), b = held(need, p);
        if (b <= a) continue;
        const size_t s0 = static_cast<size_t>(p) * plane_bytes + static_cast<size_t>(a) * row_bytes;
        const size_t s1 = static_cast<size_t>(p) * plane_bytes + static_cast<size_t>(b) * row_bytes;
        if (hi > lo && s0 == hi) {
            hi = s1;
            continue;
        }
        if (hi > lo) {
            cudaError_t e = cudaMemcpyAsync(xd + lo, xh + lo, hi - lo, cudaMemcpyHostToDevice, s);
            if (e != cudaSuccess) return e;
        }
        lo = s0;
        hi = s1;
    }
    if (hi > lo) return cudaMemcpyAsync(xd + lo, xh + lo, hi - lo, cudaMemcpyHostToDevice, s);
    return cudaSuccess;
}

// Split the m-tiles into chunks; bounds[0..n] (bounds[n] = m_tiles), returns n.
// requested > 1: that many near-equal chunks.  requested == 0: chunks of
// whole waves of units (a wave = the units the grid holds at once), so that
// splitting the launch adds no partial waves, the first one to four blocks
// long, then a ramp of short chunks, the last one block long; at most
// kMaxChunks chunks.
int plan_chunks(const Plan& P, const Geo& g, long long x_row_bytes, long long w_bytes,
                int requested, int* bounds) {
    const int MT = P.m_tiles;
    bounds[0] = 0;
    if (requested == 1 || MT < 2) {
        bounds[1] = MT;
        return 1;
    }
    if (requested > 1) {
        const int n = std::min({requested, MT, kMaxChunks});
        for (int i = 1; i <= n; ++i)
            bounds[i] = static_cast<int>(static_cast<long long>(MT) * i / n);
        return n;
    }
    const long long wave = P.grid >> P.pair;
    const long long j = wave / gcd_ll(wave, P.n_tiles);   // m-tiles per block of whole waves
    const long long nb = MT / j;
    if (nb < 2) {
        bounds[1] = MT;
        return 1;
    }
    // the first chunk (whole blocks) runs as one wave per group of column
    // tiles, each launched once its group's weights have landed: of up to
    // four blocks (two or more left for the rest), take the length whose
    // lead-in -- the input rows the chunk reads plus one weight group -- is
    // the smallest (more blocks: more waves, so smaller weight groups)
    const long long wpb = j * P.n_tiles / wave;   // waves per block
    long long b0 = 1, best = -1;
    for (long long b = 1; b <= 4 && (b == 1 || b <= nb - 2); ++b) {
        const long long wv = b * wpb;
        const long long groups =
            (wv >= 2 && wv <= kMaxWGroups && P.n_tiles % wv == 0) ? wv : 1;
        const XReach r = x_reach(g, tile_row_hi(P, static_cast<int>(b * j) - 1));
        const long long lead = r.whole * g.H * x_row_bytes +
                               (r.part - r.whole) * r.rows * x_row_bytes + w_bytes / groups;
        if (best < 0 || lead < best) {
            best = lead;
            b0 = b;
        }
    }
    // then one block (the few input rows it adds are copied right after the
    // weights, so it starts when the first chunk ends), then chunks doubling
    // up to a sixth of the rest (each one's input copied while the one
    // before runs), and one block last (a short copy-out after the last wave)
    long long blocks[kMaxChunks];
    int n = 0;
    blocks[n++] = b0;
    long long mid = nb - b0 - 1;   // blocks between the first and last chunk
    const long long share = std::max(1LL, (mid + 5) / 6);
    for (long long len = 1; mid > 0; len *= 2) {
        const long long c = n == kMaxChunks - 2 ? mid : std::min({len, share, mid});
        blocks[n++] = c;
        mid -= c;
    }
    blocks[n++] = 1;
    long long acc = 0;
    for (int i = 0; i < n; ++i) {
        acc += blocks[i] * j;
        bounds[i + 1] = static_cast<int>(acc);
    }
    bounds[n] = MT;   // the last chunk takes the m-tiles past whole blocks
    return n;
}

// Split the m-tiles into n near-equal slices of whole waves of units (a
// wave = the units the grid holds at once); bounds[0..n'], returns n'.
int plan_even_slices(const Plan& P, int n, int* bounds) {
    const long long wave = P.grid >> P.pair;
    const long long j = wave / gcd_ll(wave, P.n_tiles);   // m-tiles per block of whole waves
    const long long nb = P.m_tiles / j;
    n = static_cast<int>(std::min<long long>({static_cast<long long>(n), nb, kMaxChunks}));
    bounds[0] = 0;
    if (n < 2) {
        bounds[1] = P.m_tiles;
        return 1;
    }
    for (int i = 1; i < n; ++i) bounds[i] = static_cast<int>(nb * i / n * j);
    bounds[n] = P.m_tiles;
    return n;
}

// The slices conv_fwd_from_host runs plan P in: m-tile bounds, and the
// first slice's weight groups (gtiles column tiles each) when it spans
// several waves over all column tiles.  Point-output GEMM and split-K plans
// run unsliced.
struct SlicePlan {
    int n;
    int bounds[kMaxChunks + 1];
    int wgroups, gtiles;
};

SlicePlan plan_slices(const Plan& P, const Geo& g, int chunks) {
    SlicePlan sp;
    const long long x_row_bytes = g.W * g.C * P.elt;
    const long long w_bytes = g.K * g.T * g.R * g.S * g.C * P.elt;
    const bool chunkable = !gemm_amode(P.amode) && P.splits == 1;
    sp.bounds[0] = 0;
    sp.bounds[1] = P.m_tiles;
    sp.n = chunkable ? plan_chunks(P, g, x_row_bytes, w_bytes, chunks, sp.bounds) : 1;
    sp.wgroups = 1;
    sp.gtiles = P.n_tiles;
    if (sp.n > 1) {
        const long long wave = P.grid >> P.pair;
        const long long units0 = static_cast<long long>(sp.bounds[1] - sp.bounds[0]) * P.n_tiles;
        const long long waves0 = units0 % wave == 0 ? units0 / wave : 0;
        if (waves0 >= 2 && waves0 <= kMaxWGroups && P.n_tiles % waves0 == 0 &&
            overrides().weight_groups != 0) {
            sp.wgroups = static_cast<int>(waves0);
            sp.gtiles = P.n_tiles / sp.wgroups;
        }
    }
    return sp;
}

}  // namespace

size_t splitk_workspace_bytes(const int64_t x_dims[5], const int64_t w_dims[5],
                              const int stride[3], const int pad[3], const int dil[3], int dtype) {
    Geo g;
    DeviceInfo* d = nullptr;
    if (make_geo(x_dims, w_dims, stride, pad, dil, &g) || device_info(&d)) return 0;
    Plan P;
    if (make_plan(g, dtype, d->num_sms, d->smem_optin, SIZE_MAX, &P)) return 0;
    return P.ws_bytes - P.repack_bytes;
}

void set_last_error(const char* msg) { std::snprintf(t_last_error, sizeof t_last_error, "%s", msg); }

Overrides overrides() {
    std::lock_guard<std::mutex> lk(g_ovr_mutex);
    return g_ovr;
}

int* device_status_ptr() {
    DeviceInfo* d = nullptr;
    if (device_info(&d) != CONV_OK) return nullptr;
    return d->status;
}

}  // namespace c3d

using namespace c3d;

extern "C" {

const char* conv_last_error(void) { return t_last_error; }

const char* conv_status_string(int status) {
    switch (status) {
        case CONV_OK: return "CONV_OK";
        case CONV_ERR_INVALID: return "CONV_ERR_INVALID: invalid argument";
        case CONV_ERR_UNSUPPORTED: return "CONV_ERR_UNSUPPORTED: shape not covered by the kernels";
        case CONV_ERR_CUDA: return "CONV_ERR_CUDA: CUDA call failed";
        case CONV_ERR_TIMEOUT: return "CONV_ERR_TIMEOUT: a kernel gave up on a bounded wait";
        default: return "unknown conv_status";
    }
}

void conv_set_wait_limit_ns(uint64_t ns) { g_wait_ns = ns; }

void conv_default_overrides(conv_overrides* o) {
    if (!o) return;
    const Overrides d = {-1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1};
    std::memcpy(o, &d, sizeof d);
}

int conv_set_overrides(const conv_overrides* o) {
    Overrides v = {-1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1};
    if (o) std::memcpy(&v, o, sizeof v);
    auto in = [](int x, int lo, int hi) { return x == -1 || (x >= lo && x <= hi); };
    const bool ok =
        (v.tile_n == -1 || (v.tile_n >= 32 && v.tile_n <= 256 && v.tile_n % 32 == 0)) &&
        (v.k_bytes == -1 || v.k_bytes == 32 || v.k_bytes == 64 || v.k_bytes == 128 ||
         v.k_bytes == 256) &&
        in(v.stages, 1, 64) && in(v.group_m, 1, 1 << 20) && in(v.splits, 1, 1 << 20) &&
        in(v.pair, 0, 1) && in(v.msub, 1, 2) && in(v.slices, 1, 32) && in(v.epilogue, 1, 3) &&
        in(v.hw_major, 0, 1) && in(v.two_phase, 0, 1) && in(v.repack, 0, 1) &&
        in(v.dy_in_place, 0, 1) && in(v.pdl, 0, 1) && in(v.weight_groups, 0, 1) &&
        in(v.ncdhw_in_place, 0, 1) && (v.pack_lanes == -1 || v.pack_lanes == 2 || v.pack_lanes == 4) &&
        in(v.log, 0, 1);
    if (!ok) {
        set_error("override value out of range");
        return CONV_ERR_INVALID;
    }
    std::lock_guard<std::mutex> lk(g_ovr_mutex);
    g_ovr = v;
    return CONV_OK;
}

int conv_out_dims(const int64_t x_dims[5], const int64_t w_dims[5], const int stride[3],
                  const int pad[3], const int dil[3], int64_t out_dims[5]) {
    Geo g;
    int rc = make_geo(x_dims, w_dims, stride, pad, dil, &g);
    if (rc) return rc;
    if (!out_dims) {
        set_error("null out_dims");
        return CONV_ERR_INVALID;
    }
    out_dims[0] = g.N;
    out_dims[1] = g.Do;
    out_dims[2] = g.Ho;
    out_dims[3] = g.Wo;
    out_dims[4] = g.K;
    return CONV_OK;
}

}   // extern "C"

namespace {

// NCDHW dims [N, C, D, H, W] in the NDHWC order the geometry uses
void ndhwc_dims(const int64_t ncdhw[5], int64_t out[5]) {
    out[0] = ncdhw[0]; out[1] = ncdhw[2]; out[2] = ncdhw[3]; out[3] = ncdhw[4]; out[4] = ncdhw[1];
}

int plan_query(const Geo& g, bool ncdhw, int dtype, int num_sms, int* cls, int* tile_n,
               int* k_bytes, int* stages, int* splits, int* ctas, size_t* workspace_bytes) {
    int rc = CONV_OK;
    int sms = num_sms, smem = 232448;
    if (sms <= 0) {
        DeviceInfo* d = nullptr;
        if ((rc = device_info(&d))) return rc;
        sms = d->num_sms;
        smem = d->smem_optin;
    }
    Plan P;
    if ((rc = make_plan(g, dtype, sms, smem, SIZE_MAX, &P, ncdhw))) return rc;
    if (cls) *cls = P.cls;
    if (tile_n) *tile_n = P.BN;
    if (k_bytes) *k_bytes = P.BK;
    if (stages) *stages = P.stages;
    if (splits) *splits = P.splits;
    if (ctas) *ctas = P.grid;
    if (workspace_bytes) *workspace_bytes = P.ws_bytes;
    return CONV_OK;
}

// Patch class: the weight's rows (one patch of T*R*S*C elements each, KTRSC)
// serve as GEMM rows in place when they are already at the TMA pitch.
bool patch_weights_in_place(const Plan& P) { return P.g_row_bytes == P.tma_row_bytes; }

int fwd_impl(const Geo& g, bool ncdhw, const void* x, const void* w, int dtype,
             const float* scale_x, const float* scale_w, const float* bias, int act, void* out,
             void* workspace, size_t workspace_bytes, cudaStream_t stream);

}  // namespace

extern "C" {

int conv_fwd_plan(const int64_t x_dims[5], const int64_t w_dims[5], const int stride[3],
                  const int pad[3], const int dil[3], int dtype, int num_sms, int* cls,
                  int* tile_n, int* k_bytes, int* stages, int* splits, int* ctas,
                  size_t* workspace_bytes) {
    Geo g;
    int rc = make_geo(x_dims, w_dims, stride, pad, dil, &g);
    if (rc) return rc;
    return plan_query(g, false, dtype, num_sms, cls, tile_n, k_bytes, stages, splits, ctas,
                      workspace_bytes);
}

int conv_fwd_ncdhw_plan(const int64_t x_dims[5], const int64_t w_dims[5], const int stride[3],
                        const int pad[3], const int dil[3], int dtype, int num_sms, int* cls,
                        int* tile_n, int* k_bytes, int* stages, int* splits, int* ctas,
                        size_t* workspace_bytes) {
    if (!x_dims) {
        set_error("null shape argument");
        return CONV_ERR_INVALID;
    }
    int64_t xd[5];
    ndhwc_dims(x_dims, xd);
    Geo g;
    int rc = make_geo(xd, w_dims, stride, pad, dil, &g);
    if (rc) return rc;
    return plan_query(g, true, dtype, num_sms, cls, tile_n, k_bytes, stages, splits, ctas,
                      workspace_bytes);
}

int conv_fwd(const void* x, const int64_t x_dims[5], const void* w, const int64_t w_dims[5],
             const int stride[3], const int pad[3], const int dil[3], int dtype,
             const float* scale_x, const float* scale_w, void* out, void* workspace,
             size_t workspace_bytes, cudaStream_t stream) {
    return conv_fwd_bias(x, x_dims, w, w_dims, stride, pad, dil, dtype, scale_x, scale_w, nullptr,
                         out, workspace, workspace_bytes, stream);
}

int conv_fwd_bias(const void* x, const int64_t x_dims[5], const void* w, const int64_t w_dims[5],
                  const int stride[3], const int pad[3], const int dil[3], int dtype,
                  const float* scale_x, const float* scale_w, const float* bias, void* out,
                  void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    Geo g;
    int rc = make_geo(x_dims, w_dims, stride, pad, dil, &g);
    if (rc) return rc;
    return fwd_impl(g, false, x, w, dtype, scale_x, scale_w, bias, kActNone, out, workspace,
                    workspace_bytes, stream);
}

int conv_fwd_bias_act(const void* x, const int64_t x_dims[5], const void* w,
                      const int64_t w_dims[5], const int stride[3], const int pad[3],
                      const int dil[3], int dtype, const float* scale_x, const float* scale_w,
                      const float* bias, int act, void* out, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream) {
    Geo g;
    int rc = make_geo(x_dims, w_dims, stride, pad, dil, &g);
    if (rc) return rc;
    return fwd_impl(g, false, x, w, dtype, scale_x, scale_w, bias, act, out, workspace,
                    workspace_bytes, stream);
}

int conv_fwd_ncdhw(const void* x, const int64_t x_dims[5], const void* w, const int64_t w_dims[5],
                   const int stride[3], const int pad[3], const int dil[3], int dtype,
                   const float* scale_x, const float* scale_w, const float* bias, void* out,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!x_dims) {
        set_error("null shape argument");
        return CONV_ERR_INVALID;
    }
    int64_t xd[5];
    ndhwc_dims(x_dims, xd);
    Geo g;
    int rc = make_geo(xd, w_dims, stride, pad, dil, &g);
    if (rc) return rc;
    return fwd_impl(g, true, x, w, dtype, scale_x, scale_w, bias, kActNone, out, workspace,
                    workspace_bytes, stream);
}

}   // extern "C"

namespace {

// Launch the conv units of plan P whose kernel parameters are k (all
// m-tiles): one launch, or P.slices launches of whole waves.
cudaError_t launch_units(const Plan& P, const TMaps& tm, const KParams& k, cudaStream_t stream) {
    int bounds[kMaxChunks + 1];
    const int nsl = P.slices > 1 ? plan_even_slices(P, P.slices, bounds) : 1;
    if (nsl == 1) return launch_igemm(P.amode, P.fp8, &tm, k, P.grid, P.smem, stream);
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < nsl && e == cudaSuccess; ++i) {
        KParams ki = k;
        ki.m_tile0 = bounds[i];
        ki.m_tiles = bounds[i + 1] - bounds[i];
        const long long units = static_cast<long long>(ki.m_tiles) * P.n_tiles;
        const int grid = P.pair ? 2 * static_cast<int>(std::min<long long>(units, P.grid / 2))
                                : static_cast<int>(std::min<long long>(units, P.grid));
        e = launch_igemm(P.amode, P.fp8, &tm, ki, grid, P.smem, stream);
    }
    return e;
}

// Channel-major x through an NDHWC copy at the head of the workspace: the
// pack, then the conv of the copy, both on the caller's stream.  (Packing
// slice by slice on a second stream while the conv runs was slower, 6.9-7.2
// ms against 6.4 ms on the 3x1x1 workload: under the power cap the pack's
// draw slows the tensor-bound conv by more than the overlap saves.)
int ncdhw_via_copy(const Geo& g, const Plan& P, DeviceInfo* dev, const void* x, const void* w,
                   const float* scale_x, const float* scale_w, const float* bias, int act,
                   void* out, void* workspace, cudaStream_t stream) {
    int rc;
    void* xc = workspace;
    TMaps tm;
    if ((rc = build_maps(g, P, xc, w, &tm))) return rc;
    if ((rc = build_out_map(g, P, out, &tm))) return rc;
    KParams k;
    fill_params(g, P, xc, w, out, workspace, scale_x, scale_w, bias, dev->status, &k);
    k.act = act;
    cudaError_t e = pack_launch(x, g.N, g.C, g.D * g.H * g.W, xc, 0, nullptr, nullptr, dev, stream);
    if (e != cudaSuccess) return cuda_fail(e, "pack launch");
    if ((e = launch_units(P, tm, k, stream)) != cudaSuccess)
        return cuda_fail(e, "conv kernel launch");
    if (P.splits > 1 &&
        (e = launch_splitk_reduce(k.ws, out, P.M * g.K, P.splits, scale_x, scale_w, bias, g.K, k.act,
                                  dev->num_sms, stream)) != cudaSuccess)
        return cuda_fail(e, "split-K reduce launch");
    return CONV_OK;
}

int fwd_impl(const Geo& g, bool ncdhw, const void* x, const void* w, int dtype,
             const float* scale_x, const float* scale_w, const float* bias, int act, void* out,
             void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    int rc = CONV_OK;
    if (act < kActNone || act > kActGelu) {
        set_error("unknown activation");
        return CONV_ERR_INVALID;
    }
    if (!x || !w || !out) {
        set_error("null tensor pointer");
        return CONV_ERR_INVALID;
    }
    if (!aligned16(x) || !aligned16(w) || !aligned16(out) || (workspace && !aligned16(workspace)) ||
        (scale_x && (reinterpret_cast<uintptr_t>(scale_x) & 3u)) ||
        (scale_w && (reinterpret_cast<uintptr_t>(scale_w) & 3u)) ||
        (bias && (reinterpret_cast<uintptr_t>(bias) & 3u))) {
        set_error("device pointers must be 16-byte aligned");
        return CONV_ERR_INVALID;
    }
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev))) return rc;
    if (!load_entry_points()) {
        set_error("cuTensorMapEncode* entry points unavailable");
        return CONV_ERR_CUDA;
    }
    Plan P;
    if ((rc = make_plan(g, dtype, dev->num_sms, dev->smem_optin, workspace ? workspace_bytes : 0,
                        &P, ncdhw, act)))
        return rc;
    if (P.ncdhw_pack)
        return ncdhw_via_copy(g, P, dev, x, w, scale_x, scale_w, bias, act, out, workspace,
                              stream);
    const void* xa = x;
    const void* wa = w;
    if (P.repack == 2) {
        // the patches gathered into GEMM rows at the head of the workspace,
        // then (rows not a multiple of 16 bytes) the weights copied to the
        // same 16-byte pitch after them
        unsigned char* wsb = static_cast<unsigned char*>(workspace);
        void* wc = wsb + (P.M * P.tma_row_bytes + 255) / 256 * 256;
        // each filter row is one patch of T*R*S*C elements, already a GEMM row
        // at the TMA pitch when its bytes are a multiple of 16 (read in place),
        // else copied to that pitch by the same launch as the patches
        const bool w_in_place = patch_weights_in_place(P);
        cudaError_t e = launch_patch_gather(
            x, static_cast<int>(P.elt), g.N, g.D, g.H, g.W, g.C, static_cast<int>(g.T),
            static_cast<int>(g.R), static_cast<int>(g.S), static_cast<int>(g.Do),
            static_cast<int>(g.Ho), static_cast<int>(g.Wo), wsb, P.tma_row_bytes,
            w_in_place ? nullptr : w, g.K, wc, dev->num_sms, stream);
        if (e != cudaSuccess) return cuda_fail(e, "patch gather launch");
        xa = wsb;
        wa = w_in_place ? w : wc;
    } else if (P.repack && P.phases == 2) {
        // the two aligned weight copies (plain, shifted by 8 bytes) at the head
        // of the workspace; x is read in place
        unsigned char* wsb = static_cast<unsigned char*>(workspace);
        void* w1 = wsb + (g.K * P.tma_row_bytes + 255) / 256 * 256;
        cudaError_t e = launch_row_repack(w, wsb, g.K, w, w1, g.K, P.g_row_bytes, P.tma_row_bytes,
                                          8, dev->num_sms, stream);
        if (e != cudaSuccess) return cuda_fail(e, "row repack launch");
        wa = wsb;
    } else if (P.repack) {
        // aligned, zero-padded copies of the GEMM operands at the head of the workspace
        unsigned char* wsb = static_cast<unsigned char*>(workspace);
        void* xc = wsb;
        void* wc = wsb + (P.M * P.tma_row_bytes + 255) / 256 * 256;
        cudaError_t e = launch_row_repack(x, xc, P.M, w, wc, g.K, P.g_row_bytes, P.tma_row_bytes,
                                          0, dev->num_sms, stream);
        if (e != cudaSuccess) return cuda_fail(e, "row repack launch");
        xa = xc;
        wa = wc;
    }
    TMaps tm;
    if ((rc = build_maps(g, P, xa, wa, &tm))) return rc;
    if ((rc = build_out_map(g, P, out, &tm))) return rc;

    KParams k;
    fill_params(g, P, x, w, out, workspace, scale_x, scale_w, bias, dev->status, &k);
    k.act = act;

    if (overrides().log == 1) {
        std::fprintf(stderr,
                     "conv_fwd: class=%d amode=%d fp8=%d M=%lld K=%d BN=%d BK=%d stages=%d "
                     "splits=%d k_steps=%d tiles=%dx%d grid=%d smem=%zu tmem=%u epi=%u pair=%d msub=%d "
                     "phases=%d repack=%d\n",
                     P.cls, P.amode, P.fp8, P.M, k.K, P.BN, P.BK, P.stages, P.splits, P.k_steps,
                     P.m_tiles, P.n_tiles, P.grid, P.smem, P.tmem_cols, P.epi_bytes, P.pair, P.msub,
                     P.phases, P.repack);
    }
    cudaError_t e = launch_units(P, tm, k, stream);
    if (e != cudaSuccess) return cuda_fail(e, "conv kernel launch");
    if (P.splits > 1) {
        e = launch_splitk_reduce(k.ws, out, P.M * g.K, P.splits, scale_x, scale_w, bias, g.K, k.act,
                                 dev->num_sms, stream);
        if (e != cudaSuccess) return cuda_fail(e, "split-K reduce launch");
    }
    return CONV_OK;
}

}  // namespace

namespace {

// Workspace bytes before the kept strips of conv_fwd_ncdhw_fp8 (the amax word).
constexpr size_t kFqScratchOffset = 256;

struct FqPlan {
    FQParams p;       // geometry, tiles and shared-memory layout (pointers unset)
    int grid;
    size_t smem;
    size_t keep_bytes;   // scratch for the kept strips: grid x chunks x strip bytes
};

// The plan of conv_fwd_ncdhw_fp8: per-frame "same" filters, CTA pairs when
// the problem has two waves of 256-row units, and the strip and weight ring
// within the shared-memory budget.
int fq_plan(const Geo& g, const DeviceInfo* dev, FqPlan* fp) {
    // per-frame filters with "same" padding in H and W, unit stride and dilation
    if (g.T != 1 || g.pd != 0 || g.sd != 1 || g.sh != 1 || g.sw != 1 || g.dd != 1 || g.dh != 1 ||
        g.dw != 1 || g.R % 2 == 0 || g.S % 2 == 0 || g.ph != (g.R - 1) / 2 ||
        g.pw != (g.S - 1) / 2) {
        set_error("fused channel-major e4m3 conv: T = 1, odd R and S with pad (0, (R-1)/2, "
                  "(S-1)/2), unit stride and dilation");
        return CONV_ERR_UNSUPPORTED;
    }
    if (g.C % 16 != 0) {
        set_error("fused channel-major e4m3 conv: C must be a multiple of 16");
        return CONV_ERR_UNSUPPORTED;
    }
    if (g.H * (g.W + 2 * g.pw) > 0x3FFFFFFFll || g.N * g.D > 0x7FFFFFFFll) {
        set_error("fused channel-major e4m3 conv: frame or frame count too large");
        return CONV_ERR_UNSUPPORTED;
    }
    const Overrides ov = overrides();
    FQParams& p = fp->p;
    std::memset(&p, 0, sizeof p);
    p.N = static_cast<int>(g.N); p.C = static_cast<int>(g.C); p.D = static_cast<int>(g.D);
    p.H = static_cast<int>(g.H); p.W = static_cast<int>(g.W); p.K = static_cast<int>(g.K);
    p.R = static_cast<int>(g.R); p.S = static_cast<int>(g.S);
    p.ph = g.ph; p.pw = g.pw;
    p.Wp = p.W + 2 * p.pw;
    p.HWp = p.H * p.Wp;
    p.BN = ov.tile_n > 0 ? ov.tile_n : pick_bn(g.K);
    p.n_tiles = static_cast<int>((g.K + p.BN - 1) / p.BN);
    p.chunks = static_cast<int>((g.C + 127) / 128);
    const long long mt_pair = (p.HWp + 255) / 256;
    int pair = (g.N * g.D * mt_pair * p.n_tiles >= 2LL * dev->num_sms && dev->num_sms % 2 == 0) ? 1 : 0;
    if (ov.pair >= 0) pair = (ov.pair && dev->num_sms % 2 == 0) ? 1 : 0;
    p.pair = pair;
    p.mt_frame = (p.HWp + (128 << pair) - 1) / (128 << pair);
    const long long m_tiles = g.N * g.D * p.mt_frame;
    if (m_tiles * p.n_tiles > 0x7FFFFFFFll) {
        set_error("too many work units");
        return CONV_ERR_UNSUPPORTED;
    }
    p.m_tiles = static_cast<int>(m_tiles);
    // the strip: this CTA's 128 rows plus the taps' reach on both sides
    const long long reach = static_cast<long long>(p.ph) * p.Wp + p.pw;
    p.L = static_cast<int>((128 + 2 * reach + 31) / 32 * 32);
    p.strip_bytes = static_cast<uint32_t>(8 * p.L * 16);
    const size_t strips = (2 * static_cast<size_t>(p.strip_bytes) + 1023) / 1024 * 1024;
    const size_t staging = (static_cast<size_t>(p.strip_bytes) + 1023) / 1024 * 1024;
    const size_t fixed = 1024 + strips + staging + 160;
    // two taps per weight stage (eight MMAs per barrier round instead of
    // four: the single issuing thread spends a fixed cost per round -- wait,
    // fence, commit -- that four 128-cycle MMAs do not cover) when three such
    // stages fit; the k_bytes override forces one (128) or two (256)
    const uint32_t tap_bytes = static_cast<uint32_t>((p.BN >> pair) * 128);
    const size_t avail = static_cast<size_t>(dev->smem_optin) > fixed
                             ? static_cast<size_t>(dev->smem_optin) - fixed : 0;
    p.tap_group = (g.R * g.S >= 2 && avail / (2 * tap_bytes + 16) >= 3) ? 2 : 1;
    if (ov.k_bytes == 128) p.tap_group = 1;
    if (ov.k_bytes == 256 && g.R * g.S >= 2) p.tap_group = 2;
    p.b_stage_bytes = static_cast<uint32_t>(p.tap_group) * tap_bytes;
    if (static_cast<size_t>(dev->smem_optin) < fixed + 2 * (p.b_stage_bytes + 16)) {
        set_error("fused channel-major e4m3 conv: the filter's strip does not fit in shared "
                  "memory (frame too wide for the filter height)");
        return CONV_ERR_UNSUPPORTED;
    }
    p.b_stages = static_cast<int>(std::min<size_t>(
        8, (static_cast<size_t>(dev->smem_optin) - fixed) / (p.b_stage_bytes + 16)));
    if (ov.stages > 0) p.b_stages = std::max(2, std::min(p.b_stages, ov.stages));
    fp->smem = fixed + static_cast<size_t>(p.b_stages) * (p.b_stage_bytes + 16);
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(2 * p.BN)) cols <<= 1;
    p.tmem_cols = cols;
    p.idesc = make_idesc(1, p.BN, 128 << pair);
    // persistent CTAs (pairs) take whole m-tiles: every column tile in turn
    fp->grid = pair ? 2 * static_cast<int>(std::min<long long>(m_tiles, dev->num_sms / 2))
                    : static_cast<int>(std::min<long long>(m_tiles, dev->num_sms));
    // two scratch slots per CTA: the m-tile being copied back and the next
    p.scratch_stride = 2LL * p.chunks * p.strip_bytes;
    fp->keep_bytes = static_cast<size_t>(fp->grid) * static_cast<size_t>(p.scratch_stride);
    return CONV_OK;
}

}  // namespace

extern "C" {

int conv_fwd_from_host(const void* x_host, const int64_t x_dims[5], const void* w_host,
                       const int64_t w_dims[5], const int stride[3], const int pad[3],
                       const int dil[3], int dtype, const float* scale_x, const float* scale_w,
                       void* out_host, void* x_dev, void* w_dev, void* out_dev, void* workspace,
                       size_t workspace_bytes, int chunks, cudaStream_t stream) {
    Geo g;
    int rc = make_geo(x_dims, w_dims, stride, pad, dil, &g);
    if (rc) return rc;
    if (!x_host || !w_host || !out_host || !x_dev || !w_dev || !out_dev) {
        set_error("null tensor pointer");
        return CONV_ERR_INVALID;
    }
    if (chunks < 0) {
        set_error("chunks must be >= 0");
        return CONV_ERR_INVALID;
    }
    if (!aligned16(x_dev) || !aligned16(w_dev) || !aligned16(out_dev) ||
        (workspace && !aligned16(workspace))) {
        set_error("device pointers must be 16-byte aligned");
        return CONV_ERR_INVALID;
    }
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev))) return rc;
    if (!load_entry_points()) {
        set_error("cuTensorMapEncode* entry points unavailable");
        return CONV_ERR_CUDA;
    }
    Plan P;
    if ((rc = make_plan(g, dtype, dev->num_sms, dev->smem_optin, workspace ? workspace_bytes : 0,
                        &P)))
        return rc;
    const long long plane_bytes = g.H * g.W * g.C * P.elt;
    const size_t x_bytes = static_cast<size_t>(g.N * g.D * plane_bytes);
    const size_t x_row_bytes = static_cast<size_t>(g.W * g.C * P.elt);
    const size_t w_bytes = static_cast<size_t>(g.K * g.T * g.R * g.S * g.C * P.elt);
    const size_t row_bytes = static_cast<size_t>(g.K) * 2;   // one bf16 output row
    const unsigned char* xh = static_cast<const unsigned char*>(x_host);
    unsigned char* xd = static_cast<unsigned char*>(x_dev);
    unsigned char* oh = static_cast<unsigned char*>(out_host);
    const unsigned char* od = static_cast<const unsigned char*>(out_dev);

    const SlicePlan sp = plan_slices(P, g, chunks);
    const int n = sp.n;
    const int* bounds = sp.bounds;
    cudaError_t e;
    if (n == 1) {
        // one launch: copy in, convolve, copy out, all on the caller's stream
        if ((e = cudaMemcpyAsync(x_dev, x_host, x_bytes, cudaMemcpyHostToDevice, stream)) !=
                cudaSuccess ||
            (e = cudaMemcpyAsync(w_dev, w_host, w_bytes, cudaMemcpyHostToDevice, stream)) !=
                cudaSuccess)
            return cuda_fail(e, "cudaMemcpyAsync (host to device)");
        if ((rc = conv_fwd(x_dev, x_dims, w_dev, w_dims, stride, pad, dil, dtype, scale_x,
                           scale_w, out_dev, workspace, workspace_bytes, stream)))
            return rc;
        if ((e = cudaMemcpyAsync(out_host, out_dev, static_cast<size_t>(P.M) * row_bytes,
                                 cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
            return cuda_fail(e, "cudaMemcpyAsync (device to host)");
        return CONV_OK;
    }

    TMaps tm;
    if ((rc = build_maps(g, P, x_dev, w_dev, &tm))) return rc;
    if ((rc = build_out_map(g, P, out_dev, &tm))) return rc;
    KParams k;
    fill_params(g, P, x_dev, w_dev, out_dev, workspace, scale_x, scale_w, nullptr, dev->status,
                &k);
    k.hw_major = 0;   // slices are ranges of output rows: m-tiles in row order

    Pipe* pp = nullptr;
    if ((rc = pipe_for_device(&pp))) return rc;
    std::lock_guard<std::mutex> lk(pp->mu);
    const char* what = nullptr;
    // the copy streams start after the caller's earlier work
    if ((e = cudaEventRecord(pp->start, stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(pp->s_in, pp->start, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(pp->s_out, pp->start, 0)) != cudaSuccess)
        return cuda_fail(e, "stream ordering");
    // The first slice (whole blocks: whole waves over all column tiles) runs
    // as one wave per group of column tiles, each launched once that group's
    // weight rows have landed: the lead-in before the first kernel copies one
    // group's weights and the input rows the slice reads, not all the weights.
    const int wgroups = sp.wgroups, gtiles = sp.gtiles;
    const size_t w_row = w_bytes / static_cast<size_t>(g.K);   // one filter's bytes
    auto copy_w_group = [&](int s) -> cudaError_t {
        const long long r0 = static_cast<long long>(s) * gtiles * P.BN;
        const long long r1 = s == wgroups - 1 ? g.K : std::min<long long>(g.K, r0 + gtiles * P.BN);
        if (r1 <= r0) return cudaSuccess;
        return cudaMemcpyAsync(static_cast<unsigned char*>(w_dev) + r0 * w_row,
                               static_cast<const unsigned char*>(w_host) + r0 * w_row,
                               static_cast<size_t>(r1 - r0) * w_row, cudaMemcpyHostToDevice,
                               pp->s_in);
    };
    if ((e = copy_w_group(0)) != cudaSuccess) what = "cudaMemcpyAsync (weights)";
    // input rows on the device so far; each slice first copies the rows it
    // reads that are not there yet (the last one: everything left)
    XReach x_have{0, 0, 0};
    for (int i = 0; i < n && !what; ++i) {
        const int mt0 = bounds[i], mt1 = bounds[i + 1];
        const long long row_lo = tile_row_lo(P, mt0), row_hi = tile_row_hi(P, mt1 - 1);
        const XReach x_need =
            i == n - 1 ? XReach{g.N * g.D, g.N * g.D, 0} : x_reach(g, row_hi);
        if ((e = copy_x_reach(g, x_have, x_need, static_cast<size_t>(plane_bytes), x_row_bytes,
                              xh, xd, pp->s_in)) != cudaSuccess) {
            what = "cudaMemcpyAsync (activation)";
            break;
        }
        x_have = x_need;
        if ((e = cudaEventRecord(pp->ev_in[i], pp->s_in)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(stream, pp->ev_in[i], 0)) != cudaSuccess) {
            what = "stream ordering";
            break;
        }
        // the other weight groups follow the first slice's input planes
        for (int s = 1; i == 0 && s < wgroups && !what; ++s)
            if ((e = copy_w_group(s)) != cudaSuccess ||
                (e = cudaEventRecord(pp->ev_w[s], pp->s_in)) != cudaSuccess)
                what = "cudaMemcpyAsync (weights)";
        if (what) break;
        k.m_tile0 = mt0;
        k.m_tiles = mt1 - mt0;
        const int parts = i == 0 ? wgroups : 1;
        for (int s = 0; s < parts && !what; ++s) {
            k.n_tile0 = parts > 1 ? s * gtiles : 0;
            k.n_tiles = parts > 1 ? gtiles : P.n_tiles;
            if (s > 0 && (e = cudaStreamWaitEvent(stream, pp->ev_w[s], 0)) != cudaSuccess) {
                what = "stream ordering";
                break;
            }
            const long long units = static_cast<long long>(k.m_tiles) * k.n_tiles;
            const int grid = P.pair ? 2 * static_cast<int>(std::min<long long>(units, P.grid / 2))
                                    : static_cast<int>(std::min<long long>(units, P.grid));
            if (overrides().log == 1)
                std::fprintf(stderr, "conv_fwd_from_host: chunk %d m-tiles [%d, %d) n-tiles "
                             "[%d, %d) rows [%lld, %lld) x planes %lld whole + %lld rows of "
                             "[%lld, %lld) grid %d\n", i, mt0, mt1, k.n_tile0,
                             k.n_tile0 + k.n_tiles, row_lo, row_hi, x_have.whole, x_have.rows,
                             x_have.whole, x_have.part, grid);
            if ((e = launch_igemm(P.amode, P.fp8, &tm, k, grid, P.smem, stream)) != cudaSuccess)
                what = "conv kernel launch";
        }
        k.n_tile0 = 0;
        k.n_tiles = P.n_tiles;
        if (what) break;
        if ((e = cudaEventRecord(pp->ev_conv[i], stream)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(pp->s_out, pp->ev_conv[i], 0)) != cudaSuccess) {
            what = "stream ordering";
            break;
        }
        if ((e = cudaMemcpyAsync(oh + row_lo * row_bytes, od + row_lo * row_bytes,
                                 static_cast<size_t>(row_hi - row_lo) * row_bytes,
                                 cudaMemcpyDeviceToHost, pp->s_out)) != cudaSuccess) {
            what = "cudaMemcpyAsync (output)";
            break;
        }
    }
    // the caller's stream continues after both copy streams, also on failure
    cudaError_t e2;
    if ((e2 = cudaEventRecord(pp->in_done, pp->s_in)) != cudaSuccess ||
        (e2 = cudaEventRecord(pp->out_done, pp->s_out)) != cudaSuccess ||
        (e2 = cudaStreamWaitEvent(stream, pp->in_done, 0)) != cudaSuccess ||
        (e2 = cudaStreamWaitEvent(stream, pp->out_done, 0)) != cudaSuccess) {
        if (!what) return cuda_fail(e2, "stream ordering");
    }
    if (what) return cuda_fail(e, what);
    return CONV_OK;
}

int conv_fwd_from_host_slices(const int64_t x_dims[5], const int64_t w_dims[5],
                              const int stride[3], const int pad[3], const int dil[3], int dtype,
                              int num_sms, size_t workspace_bytes, int chunks, int* n_slices,
                              int64_t* rows, int64_t* reach, int* weight_groups) {
    Geo g;
    int rc = make_geo(x_dims, w_dims, stride, pad, dil, &g);
    if (rc) return rc;
    if (!n_slices || !rows || !reach || !weight_groups) {
        set_error("null output pointer");
        return CONV_ERR_INVALID;
    }
    if (chunks < 0) {
        set_error("chunks must be >= 0");
        return CONV_ERR_INVALID;
    }
    int sms = num_sms, smem = 232448;
    if (sms <= 0) {
        DeviceInfo* d = nullptr;
        if ((rc = device_info(&d))) return rc;
        sms = d->num_sms;
        smem = d->smem_optin;
    }
    Plan P;
    if ((rc = make_plan(g, dtype, sms, smem, workspace_bytes, &P))) return rc;
    const SlicePlan sp = plan_slices(P, g, chunks);
    *n_slices = sp.n;
    *weight_groups = sp.wgroups;
    for (int i = 0; i < sp.n; ++i) {
        const long long lo = sp.n == 1 ? 0 : tile_row_lo(P, sp.bounds[i]);
        const long long hi = sp.n == 1 ? P.M : tile_row_hi(P, sp.bounds[i + 1] - 1);
        const XReach r = i == sp.n - 1 ? XReach{g.N * g.D, g.N * g.D, 0} : x_reach(g, hi);
        rows[2 * i] = lo;
        rows[2 * i + 1] = hi;
        reach[3 * i] = r.whole;
        reach[3 * i + 1] = r.part;
        reach[3 * i + 2] = r.rows;
    }
    return CONV_OK;
}

int pack_ncdhw_bf16_to_ndhwc(const void* in, const int64_t dims[5], void* out,
                             cudaStream_t stream) {
    if (!in || !out || !dims) {
        set_error("null argument");
        return CONV_ERR_INVALID;
    }
    for (int i = 0; i < 5; ++i)
        if (dims[i] <= 0) {
            set_error("dims must be positive");
            return CONV_ERR_INVALID;
        }
    if (!aligned16(in) || !aligned16(out)) {
        set_error("device pointers must be 16-byte aligned");
        return CONV_ERR_INVALID;
    }
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc) return rc;
    const long long S = dims[2] * dims[3] * dims[4];
    cudaError_t e = pack_launch(in, dims[0], dims[1], S, out, 0, nullptr, nullptr, dev, stream);
    if (e != cudaSuccess) return cuda_fail(e, "pack launch");
    return CONV_OK;
}

size_t pack_fp8_workspace_size(void) { return 16; }

int pack_ncdhw_bf16_to_ndhwc_fp8(const void* in, const int64_t dims[5], void* out,
                                 float* scale_out, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream) {
    if (!in || !out || !dims || !scale_out || !workspace) {
        set_error("null argument");
        return CONV_ERR_INVALID;
    }
    if (workspace_bytes < pack_fp8_workspace_size()) {
        set_error("workspace too small");
        return CONV_ERR_INVALID;
    }
    for (int i = 0; i < 5; ++i)
        if (dims[i] <= 0) {
            set_error("dims must be positive");
            return CONV_ERR_INVALID;
        }
    if (!aligned16(in) || !aligned16(out) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(scale_out) & 3u)) {
        set_error("device pointers must be 16-byte aligned");
        return CONV_ERR_INVALID;
    }
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc) return rc;
    const long long S = dims[2] * dims[3] * dims[4];
    const long long n = dims[0] * dims[1] * S;
    unsigned int* amax = static_cast<unsigned int*>(workspace);
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(unsigned int), stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    e = launch_amax_bf16(in, n, amax, dev->num_sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "amax launch");
    e = pack_launch(in, dims[0], dims[1], S, out, 1, amax, scale_out, dev, stream);
    if (e != cudaSuccess) return cuda_fail(e, "pack launch");
    return CONV_OK;
}

int conv_fwd_kernel_launches(const int64_t x_dims[5], const int64_t w_dims[5],
                             const int stride[3], const int pad[3], const int dil[3], int dtype,
                             size_t workspace_bytes, int* launches) {
    Geo g;
    int rc = make_geo(x_dims, w_dims, stride, pad, dil, &g);
    if (rc) return rc;
    if (!launches) {
        set_error("null argument");
        return CONV_ERR_INVALID;
    }
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev))) return rc;
    Plan P;
    if ((rc = make_plan(g, dtype, dev->num_sms, dev->smem_optin, workspace_bytes, &P))) return rc;
    int n = P.repack ? 1 : 0;
    if (P.repack == 2)   // the patch gather, with the weights' copy unless read in place
        n = patch_gather_launches(static_cast<int>(P.elt), g.N, g.D, g.H, g.W, g.C,
                                  static_cast<int>(g.T), static_cast<int>(g.R),
                                  static_cast<int>(g.S), static_cast<int>(g.Do),
                                  static_cast<int>(g.Ho), static_cast<int>(g.Wo), P.tma_row_bytes,
                                  !patch_weights_in_place(P), g.K);
    int bounds[kMaxChunks + 1];
    n += P.slices > 1 ? plan_even_slices(P, P.slices, bounds) : 1;
    if (P.splits > 1) ++n;
    *launches = n;
    return CONV_OK;
}

int conv_bwd_point_workspace_bytes(const int64_t x_dims[5], const int64_t w_dims[5],
                                   const int stride[3], const int pad[3], const int dil[3],
                                   int which, size_t* bytes) {
    Geo g;
    int rc = make_geo(x_dims, w_dims, stride, pad, dil, &g);
    if (rc) return rc;
    if (!bytes || (which != 0 && which != 1)) {
        set_error("bytes must be non-NULL and which 0 (data) or 1 (weights)");
        return CONV_ERR_INVALID;
    }
    if (!is_point_output(g)) {
        set_error("backward passes cover point-output shapes only");
        return CONV_ERR_UNSUPPORTED;
    }
    const long long N = g.N, K = g.K, J = g.T * g.R * g.S * g.C;
    const int one[3] = {1, 1, 1}, zero[3] = {0, 0, 0};
    size_t inner = 0, head;
    if (which == 0) {
        const int64_t xi[5] = {N, 1, 1, 1, K}, wi[5] = {J, 1, 1, 1, K};
        head = round256(J * K * 2);
        rc = conv_fwd_plan(xi, wi, one, zero, one, CONV_DTYPE_BF16, 0, nullptr, nullptr, nullptr,
                           nullptr, nullptr, nullptr, &inner);
    } else {
        const long long Np = (N + 7) / 8 * 8;
        const int64_t xi[5] = {K, 1, 1, 1, Np}, wi[5] = {J, 1, 1, 1, Np};
        head = round256(K * Np * 2) + round256(J * Np * 2);
        rc = conv_fwd_plan(xi, wi, one, zero, one, CONV_DTYPE_BF16, 0, nullptr, nullptr, nullptr,
                           nullptr, nullptr, nullptr, &inner);
    }
    if (rc) return rc;
    *bytes = head + inner;
    return CONV_OK;
}

int conv_bwd_data_point(const void* dy, const void* w, const int64_t x_dims[5],
                        const int64_t w_dims[5], const int stride[3], const int pad[3],
                        const int dil[3], void* dx, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
    long long N, K, J;
    int rc = bwd_setup(x_dims, w_dims, stride, pad, dil, dy, w, dx, workspace, &N, &K, &J);
    if (rc) return rc;
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev))) return rc;
    const size_t head = round256(J * K * 2);
    if (!workspace || workspace_bytes < head) {
        set_error("workspace smaller than the transposed weights (see conv_bwd_point_workspace_bytes)");
        return CONV_ERR_INVALID;
    }
    // w [K, J] -> w^T [J, K]: the GEMM dx[N, J] = dy[N, K] w[K, J] then has
    // both operands K-major, and is the pointwise forward conv of dy by w^T
    cudaError_t e = launch_transpose_pad(w, K, J, workspace, K, dev->num_sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "transpose launch");
    const int64_t xi[5] = {N, 1, 1, 1, K}, wi[5] = {J, 1, 1, 1, K};
    const int one[3] = {1, 1, 1}, zero[3] = {0, 0, 0};
    return conv_fwd(dy, xi, workspace, wi, one, zero, one, CONV_DTYPE_BF16, nullptr, nullptr, dx,
                    static_cast<unsigned char*>(workspace) + head, workspace_bytes - head, stream);
}

int conv_bwd_weight_point(const void* x, const void* dy, const int64_t x_dims[5],
                          const int64_t w_dims[5], const int stride[3], const int pad[3],
                          const int dil[3], void* dw, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
    long long N, K, J;
    int rc = bwd_setup(x_dims, w_dims, stride, pad, dil, x, dy, dw, workspace, &N, &K, &J);
    if (rc) return rc;
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev))) return rc;
    // the reduction runs over the batch: dy^T [K, Np] and x^T [J, Np], rows
    // zero-padded to Np (a multiple of 8 elements, 16 bytes)
    const long long Np = (N + 7) / 8 * 8;
    if (K % 8 == 0 && overrides().dy_in_place != 0) {
        // dy's rows are 16-byte multiples: the GEMM reads dy in place as an
        // MN-major A; only x is transposed
        const size_t head = round256(J * Np * 2);
        if (workspace && workspace_bytes >= head) {
            unsigned char* wsb = static_cast<unsigned char*>(workspace);
            cudaError_t e = launch_transpose_pad(x, N, J, wsb, Np, dev->num_sms, stream);
            if (e != cudaSuccess) return cuda_fail(e, "transpose launch");
            rc = gemm_mn_a(dy, K, N, wsb, J, Np, dw, wsb + head, workspace_bytes - head, dev,
                           stream);
            if (rc != CONV_ERR_UNSUPPORTED) return rc;
        }
    }
    const size_t dyt = round256(K * Np * 2), head = dyt + round256(J * Np * 2);
    if (!workspace || workspace_bytes < head) {
        set_error("workspace smaller than the transposed operands (see conv_bwd_point_workspace_bytes)");
        return CONV_ERR_INVALID;
    }
    unsigned char* wsb = static_cast<unsigned char*>(workspace);
    cudaError_t e = launch_transpose_pad(dy, N, K, wsb, Np, dev->num_sms, stream);
    if (e == cudaSuccess) e = launch_transpose_pad(x, N, J, wsb + dyt, Np, dev->num_sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "transpose launch");
    const int64_t xi[5] = {K, 1, 1, 1, Np}, wi[5] = {J, 1, 1, 1, Np};
    const int one[3] = {1, 1, 1}, zero[3] = {0, 0, 0};
    return conv_fwd(wsb, xi, wsb + dyt, wi, one, zero, one, CONV_DTYPE_BF16, nullptr, nullptr, dw,
                    wsb + head, workspace_bytes - head, stream);
}

size_t conv_fwd_workspace_size(const int64_t x_dims[5], const int64_t w_dims[5],
                               const int stride[3], const int pad[3], const int dil[3],
                               int dtype) {
    size_t bytes = 0;
    if (conv_fwd_plan(x_dims, w_dims, stride, pad, dil, dtype, 0, nullptr, nullptr, nullptr,
                      nullptr, nullptr, nullptr, &bytes) != CONV_OK)
        return 0;
    return bytes;
}

int conv_fwd_ncdhw_fp8_workspace_size(const int64_t x_dims[5], const int64_t w_dims[5],
                                      const int stride[3], const int pad[3], const int dil[3],
                                      size_t* bytes) {
    if (!x_dims || !bytes) {
        set_error("null argument");
        return CONV_ERR_INVALID;
    }
    int64_t xd[5];
    ndhwc_dims(x_dims, xd);
    Geo g;
    int rc = make_geo(xd, w_dims, stride, pad, dil, &g);
    if (rc) return rc;
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev))) return rc;
    FqPlan fp;
    if ((rc = fq_plan(g, dev, &fp))) return rc;
    *bytes = kFqScratchOffset + fp.keep_bytes;
    return CONV_OK;
}

int conv_fwd_ncdhw_fp8(const void* x, const int64_t x_dims[5], const void* w,
                       const int64_t w_dims[5], const int stride[3], const int pad[3],
                       const int dil[3], const float* scale_w, float* scale_x_out,
                       const float* bias, void* out, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream) {
    if (!x_dims) {
        set_error("null shape argument");
        return CONV_ERR_INVALID;
    }
    int64_t xd[5];
    ndhwc_dims(x_dims, xd);
    Geo g;
    int rc = make_geo(xd, w_dims, stride, pad, dil, &g);
    if (rc) return rc;
    if (!x || !w || !out || !workspace) {
        set_error("null tensor or workspace pointer");
        return CONV_ERR_INVALID;
    }
    if (workspace_bytes < pack_fp8_workspace_size()) {
        set_error("workspace smaller than pack_fp8_workspace_size()");
        return CONV_ERR_INVALID;
    }
    if (!aligned16(x) || !aligned16(w) || !aligned16(out) || !aligned16(workspace) ||
        (scale_w && (reinterpret_cast<uintptr_t>(scale_w) & 3u)) ||
        (scale_x_out && (reinterpret_cast<uintptr_t>(scale_x_out) & 3u)) ||
        (bias && (reinterpret_cast<uintptr_t>(bias) & 3u))) {
        set_error("device pointers must be 16-byte aligned");
        return CONV_ERR_INVALID;
    }
    DeviceInfo* dev = nullptr;
    if ((rc = device_info(&dev))) return rc;
    if (!load_entry_points()) {
        set_error("cuTensorMapEncode* entry points unavailable");
        return CONV_ERR_CUDA;
    }
    FqPlan fp;
    if ((rc = fq_plan(g, dev, &fp))) return rc;
    FQParams& p = fp.p;
    unsigned int* amax = static_cast<unsigned int*>(workspace);
    // with room after the amax word, the converters work one m-tile ahead into
    // a scratch there and every column tile copies the strips back
    if (workspace_bytes >= kFqScratchOffset + fp.keep_bytes)
        p.scratch = static_cast<unsigned char*>(workspace) + kFqScratchOffset;
    p.x = static_cast<const unsigned short*>(x);
    p.amax_bits = amax;
    p.scale_x_out = scale_x_out;
    p.scale_w = scale_w;
    p.bias = bias;
    p.out = out;
    p.status = dev->status;
    p.wait_ns = g_wait_ns;
    // the e4m3 weight [K, R*S, C] as {C, K, R*S}: boxes of 128 channel bytes x
    // (BN >> pair) filters x tap_group taps, 128-byte swizzle, so a stage is
    // tap_group blocks of (BN >> pair) rows x 128 bytes (taps past R*S, in the
    // last group of an odd count, read as zeros)
    CUtensorMap wm;
    {
        const cuuint64_t taps = static_cast<cuuint64_t>(g.R * g.S);
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(g.C), static_cast<cuuint64_t>(g.K), taps};
        const cuuint64_t str[2] = {static_cast<cuuint64_t>(g.C) * taps, static_cast<cuuint64_t>(g.C)};
        const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(p.BN >> p.pair),
                                   static_cast<cuuint32_t>(p.tap_group)};
        if ((rc = encode_tiled(&wm, 1, 3, w, dims, str, box, 128))) return rc;
    }
    if (overrides().log == 1)
        std::fprintf(stderr, "conv_fwd_ncdhw_fp8: BN=%d pair=%d L=%d strip=%u b_stages=%d "
                     "tap_group=%d m_tiles=%d n_tiles=%d chunks=%d grid=%d smem=%zu keep=%d\n",
                     p.BN, p.pair, p.L, p.strip_bytes, p.b_stages, p.tap_group, p.m_tiles,
                     p.n_tiles, p.chunks, fp.grid, fp.smem, p.scratch ? 1 : 0);
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(unsigned int), stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    e = launch_amax_bf16(x, g.N * g.C * g.D * g.H * g.W, amax, dev->num_sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "amax launch");
    e = launch_fused_q(&wm, p, fp.grid, fp.smem, stream);
    if (e != cudaSuccess) return cuda_fail(e, "fused conv launch");
    return CONV_OK;
}

int conv_get_device_status_stream(cudaStream_t stream, int* device_status) {
    if (!device_status) {
        set_error("null argument");
        return CONV_ERR_INVALID;
    }
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc) return rc;
    // read, then clear, in stream order after the stream's earlier work
    int v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, dev->status, sizeof v, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(dev->status, 0, sizeof(int), stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "status read on the stream");
    *device_status = v;
    return CONV_OK;
}

int conv_get_device_status(int* device_status) {
    if (!device_status) {
        set_error("null argument");
        return CONV_ERR_INVALID;
    }
    DeviceInfo* dev = nullptr;
    int rc = device_info(&dev);
    if (rc) return rc;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof v);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol");
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol");
    *device_status = v;
    return CONV_OK;
}

}  // extern "C"
