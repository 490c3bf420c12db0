// internal.h -- parameter blocks and launch entry points shared by the host
// library (conv3d_api.cu) and the kernel translation units.  Not part of the
// public ABI.
#pragma once
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace c3d {

// How the A operand (the implicit im2col matrix) reaches shared memory.
enum AMode : int {
    AM_IM2COL = 0,     // TMA im2col-mode box per (tap, channel chunk)
    AM_TEMPORAL = 1,   // T x 1 x 1 filter: one TMA tiled 4-D box of HW rows
    AM_GEMM_TMA = 2,   // plain GEMM, 16-byte aligned rows: TMA tiled 2-D boxes
    AM_GEMM_GATHER = 3 // plain GEMM, rows not 16-byte aligned: cp.async gather
};

constexpr int kBM = 128;               // rows of a tile (tcgen05 M, one CTA)
constexpr int kEpiWarps = 4;           // warps reading TMEM in the epilogue
// epilogue activations (values of conv_fwd_bias_act's `act`)
constexpr int kActNone = 0, kActRelu = 1, kActSilu = 2, kActGelu = 3;

// 1/x by the approximate reciprocal instruction (about 1 ulp; 1/inf = 0):
// the epilogue's activations feed bf16 outputs, far coarser than that.
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// erf(x) by Abramowitz & Stegun, Handbook of Mathematical Functions, formula
// 7.1.26: 1 - (a1 t + ... + a5 t^5) e^(-x^2), t = 1 / (1 + p x) for x >= 0,
// odd in x; |error| <= 1.5e-7, far below the bf16 output's resolution, at a
// fraction of the cost of a full-precision erf in an epilogue that has one
// evaluation per output element.
__device__ __forceinline__ float erf_as7126(float x) {
    const float a = fabsf(x);
    const float t = rcp_approx(fmaf(0.3275911f, a, 1.0f));
    const float poly =
        t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, 1.061405429f, -1.453152027f), 1.421413741f),
                         -0.284496736f),
                 0.254829592f);
    return copysignf(1.0f - poly * __expf(-a * a), x);
}

// The activation on an fp32 epilogue value: max(v, 0); v * sigmoid(v);
// v * Phi(v) = v/2 * (1 + erf(v / sqrt(2))), the erf form of GELU.
template <int ACT>
__device__ __forceinline__ float activate_c(float v) {
    if constexpr (ACT == kActRelu) return fmaxf(v, 0.0f);
    else if constexpr (ACT == kActSilu) return v * rcp_approx(1.0f + __expf(-v));
    else if constexpr (ACT == kActGelu)
        return 0.5f * v * (1.0f + erf_as7126(v * 0.70710678118654752f));
    else return v;
}

__device__ __forceinline__ float activate(float v, int act) {
    if (act == kActRelu) return activate_c<kActRelu>(v);
    if (act == kActSilu) return activate_c<kActSilu>(v);
    if (act == kActGelu) return activate_c<kActGelu>(v);
    return v;
}
constexpr int kGatherThreads = 128;    // producer threads of AM_GEMM_GATHER
constexpr uint32_t kEpiChunkBytes = 32 * 32 * 2;              // one warp's 32x32 bf16 chunk
constexpr uint32_t kEpiStageBytes = kEpiWarps * 2 * kEpiChunkBytes;   // double-buffered

// Division by a launch constant d (1 <= d <= 2^31) as a multiply-high, an add
// and a shift (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994, section 4): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, floor(x / d) = (umulhi(x, m) + x) >> l for
// every 32-bit x, the sum taken in 33 bits.  The kernels' per-unit index
// arithmetic (unit -> tile, row -> output position, k-step -> tap) divides
// by these instead of issuing integer divisions.
struct FastDiv {
    uint32_t d, mul, shift;
};

inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f{d < 1u ? 1u : d, 1u, 0u};
    while ((1ull << f.shift) < f.d) ++f.shift;
    f.mul = static_cast<uint32_t>((((1ull << 32) * ((1ull << f.shift) - f.d)) / f.d) + 1ull);
    return f;
}

__device__ __forceinline__ uint32_t fdiv(uint32_t x, const FastDiv& f) {
    return static_cast<uint32_t>((static_cast<uint64_t>(__umulhi(x, f.mul)) + x) >> f.shift);
}

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) only when this kernel has
// not yet been allowed `smem` bytes on the current device: `slots` (one per
// kernel, static in its launcher) remembers the largest size set on each
// device, so repeated launches (22 per call on long reductions) skip the
// driver call.  The attribute belongs to the device context, so a
// cudaDeviceReset invalidates it like the library's other per-device state.
constexpr int kMaxDevices = 64;
template <typename Kernel>
cudaError_t ensure_dynamic_smem(Kernel kern, size_t smem, std::atomic<int>* slots) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int want = static_cast<int>(smem);
    if (dev >= 0 && dev < kMaxDevices && slots[dev].load(std::memory_order_acquire) >= want)
        return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
    if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
        int cur = slots[dev].load(std::memory_order_relaxed);
        while (cur < want && !slots[dev].compare_exchange_weak(cur, want, std::memory_order_acq_rel)) {
        }
    }
    return e;
}

struct KParams {
    // convolution geometry (A coordinates)
    int N, D, H, W, C;
    int T, R, S;
    int Do, Ho, Wo;
    int sd, sh, sw, pd, ph, pw, dd, dh, dw;
    // GEMM view
    long long M;        // output rows
    int K;              // output columns (filters)
    int HW;             // temporal: H*W rows per (n, d) plane
    int hw_tiles;       // temporal: ceil(HW / rows per m-tile)
    int hw_major;       // temporal: m-tiles ordered H*W tile major (see temporal_tile)
    int m_tiles, n_tiles, splits;
    int m_tile0;        // first m-tile of this launch (launches over a range of m-tiles)
    // row phases of the point-output GEMM (1, or 2 when every other A row is
    // not 16-byte aligned): output row = local row * phases + phase; m-tiles
    // [0, mt_phase0) are phase 0, the rest phase 1; rows0 / rows1 rows each
    int phases, mt_phase0;
    long long rows0, rows1;
    int k_steps;        // k-steps of the whole reduction
    int steps_per_split;
    int taps;           // conv: T*R*S
    int group_m;        // raster: consecutive m-tiles per group
    // tile / pipeline shape (runtime)
    int BN;             // tile columns, multiple of 32, <= 256
    int BK;             // bytes of one row per k-step: 32, 64, 128 or 256
    int stages;
    uint32_t a_stage_bytes, b_stage_bytes, stage_bytes;
    uint32_t idesc;     // tcgen05 instruction descriptor
    uint32_t layout;    // smem descriptor swizzle code
    uint32_t sbo;       // smem descriptor stride byte offset (8 rows)
    uint32_t tmem_cols; // allocated TMEM columns (power of two >= 2*BN)
    uint32_t epi_bytes; // shared staging of the epilogue (0: direct stores from registers)
    int epi_mode;       // 0 direct stores, 1 TMA tensor stores, 2 staged 8- / 4-byte stores
    int pair;           // 1: CTA-pair kernel (cluster of 2, 256-row units)
    int a_mn;           // 1: A is MN-major in memory (M contiguous; 128- or 256-byte k-steps):
                        //    GEMM mode [K rows, M], or temporal mode over channel-major x
    int msub;           // row sub-tiles per unit sharing each B stage (1 or 2)
    int n_tile0;        // first column tile of this launch (n_tiles column tiles from it)
    int act;            // activation after scale and bias: kActNone / Relu / Silu / Gelu
    // AM_GEMM_GATHER operands: A [M, g_cols], B [K, g_cols] row-major
    const unsigned char* ga;
    const unsigned char* gb;
    long long g_row_bytes;
    // outputs
    void* out;          // bf16 [M, K]
    float* ws;          // split-K partials [splits, M, K]
    const float* scale_x;
    const float* scale_w;
    const float* bias;  // fp32 [K] added after the scales, or NULL
    int* status;        // device status word
    unsigned long long wait_ns;
    // divisors of the per-unit index arithmetic, filled at launch from the
    // fields above (set_divisors): units per split, units per raster group,
    // group_m, temporal planes (N * Do) and H*W tiles, Do, Ho, Wo, taps, S, R;
    // rows32: every row index (plus a tile) fits in 31 bits
    FastDiv f_tiles, f_group, f_gm, f_planes, f_hw_tiles, f_Do, f_Ho, f_Wo, f_taps, f_S, f_R;
    int rows32;
};

// The tensor maps of one launch: A, B and the output for each row phase
// (index 1 is used only by a two-phase point-output GEMM).
struct TMaps {
    CUtensorMap a[2], b[2], c[2];
};

// Parameters of the fused channel-major e4m3 convolution (conv_fused_q.cu):
// bf16 x NCDHW read in place and quantised while the A operand is built.
// Output rows are enumerated in padded-row coordinates: per (n, d) frame,
// P = h * Wp + wp with Wp = W + 2*pw, image column w = wp - pw (rows with
// wp outside [pw, pw + W) are computed and dropped).  Each CTA's 128 rows
// read a strip of L padded positions around them; tap (r, s) is the strip
// shifted by r*Wp + s positions.
struct FQParams {
    int N, C, D, H, W, K, R, S, ph, pw;
    int Wp, HWp;          // padded row length, padded positions per frame
    int mt_frame;         // m-tiles per frame (128 << pair rows each)
    int m_tiles, n_tiles; // m_tiles = N * D * mt_frame
    int chunks;           // ceil(C / 128): 128-channel reduction chunks
    int BN;               // tile columns (multiple of 32, <= 256)
    int b_stages;         // weight ring depth
    int tap_group;        // filter taps per weight stage (1 or 2): one barrier round each
    int L;                // strip positions per CTA (multiple of 32)
    uint32_t strip_bytes; // 8 slices x L x 16 bytes
    uint32_t b_stage_bytes; // tap_group x (BN >> pair) x 128 bytes
    uint32_t idesc;       // tcgen05 instruction descriptor (e4m3 x e4m3, M, N)
    uint32_t tmem_cols;
    int pair;
    unsigned char* scratch;        // per-CTA converted strips (blockIdx.x * scratch_stride), or NULL
    long long scratch_stride;      // 2 slots x chunks x strip_bytes
    const unsigned short* x;       // bf16 NCDHW
    const unsigned int* amax_bits; // max |x| as binary32 bits (computed before)
    float* scale_x_out;            // receives amax / 448 (or NULL)
    const float* scale_w;
    const float* bias;
    void* out;                     // bf16 NDHWC
    int* status;
    unsigned long long wait_ns;
};
constexpr int kFqThreads = 480;   // warp 0 weights (TMA), 1 MMA, 2-5 epilogue, 6 strip loader,
                                  // 7-14 converters

// Launch the fused channel-major e4m3 convolution (w_map: the e4m3 KTRSC
// weight as {C, K, R*S} with boxes {128, BN >> pair, tap_group}, 128-byte
// swizzle: a stage holds tap_group consecutive taps' filter rows, one
// (BN >> pair) x 128-byte block per tap).
cudaError_t launch_fused_q(const CUtensorMap* w_map, const FQParams& p, int grid, size_t smem,
                           cudaStream_t stream);

// Launch the implicit-GEMM kernel (AMODE x dtype) on grid/smem from the plan.
cudaError_t launch_igemm(int amode, int fp8, const TMaps* maps, const KParams& p, int grid,
                         size_t smem, cudaStream_t stream);

// Deterministic split-K reduction: out = bf16(act(scale * sum_s ws[s] + bias[k]))
// in split order (bias may be NULL; k = column of the [M, K] output).
cudaError_t launch_splitk_reduce(const float* ws, void* out, long long MK, int splits,
                                 const float* scale_x, const float* scale_w, const float* bias,
                                 long long K, int act, int num_sms, cudaStream_t stream);

// Row repack of two matrices with equal row pitches: copy rows of
// src_row_bytes into rows of dst_row_bytes, matrix 1's rows shifted right by
// dst1_shift_bytes, zero-filling the rest of each destination row.
cudaError_t launch_row_repack(const void* src0, void* dst0, long long rows0, const void* src1,
                              void* dst1, long long rows1, long long src_row_bytes,
                              long long dst_row_bytes, long long dst1_shift_bytes, int num_sms,
                              cudaStream_t stream);

// Patch gather of a stride == filter convolution: row (n, od, oh, ow) of `a`
// (pitch_bytes per row, tail zeroed) is the patch's T*R*S*C elements.  With
// w != NULL, the K filter rows of w (T*R*S*C elements each) are copied to
// `wc` at the same pitch too, in the same launch when the word counts allow.
cudaError_t launch_patch_gather(const void* x, int elt, long long N, long long D, long long H,
                                long long W, long long C, int T, int R, int S, int Do, int Ho,
                                int Wo, void* a, long long pitch_bytes, const void* w,
                                long long K, void* wc, int num_sms, cudaStream_t stream);
// Kernel launches launch_patch_gather makes for that problem (1 or 2).
int patch_gather_launches(int elt, long long N, long long D, long long H, long long W, long long C,
                          int T, int R, int S, int Do, int Ho, int Wo, long long pitch_bytes,
                          bool with_w, long long K);

// 16-bit transpose: dst[c, r] = src[r, c] for src [R, C] dense, dst rows of
// P >= R elements with [R, P) zero-filled.
cudaError_t launch_transpose_pad(const void* src, long long R, long long C, void* dst,
                                 long long P, int num_sms, cudaStream_t stream);

// Bytes of split-K partials the plan for this problem uses (0 without split-K).
size_t splitk_workspace_bytes(const int64_t x_dims[5], const int64_t w_dims[5],
                              const int stride[3], const int pad[3], const int dil[3], int dtype);

// Pack kernels.
cudaError_t launch_amax_bf16(const void* in, long long n, unsigned int* amax_bits, int num_sms,
                             cudaStream_t stream);
cudaError_t launch_pack(const void* in, long long N, long long C, long long S, void* out,
                        int fp8, const unsigned int* amax_bits, float* scale_out, int num_sms,
                        cudaStream_t stream);

// TMA-fed pack (C % 8 == 0, S % 8 == 0): in_map is the bf16 input as a 3-D
// tensor {S, C, N} with a box of {256, 128, 1} and no swizzle.  pack_tma_stages gives the shared-memory ring depth for the
// device's per-block limit (0: the kernel does not fit).
int pack_tma_stages(int fp8, int smem_optin);
cudaError_t launch_pack_tma(const CUtensorMap* in_map, long long N, long long C, long long S,
                            void* out, int fp8, const unsigned int* amax_bits, float* scale_out,
                            int num_sms, int smem_optin, int* status, unsigned long long wait_ns,
                            cudaStream_t stream);

int* device_status_ptr();   // device address of the status word (current device)

// The process's plan / path overrides (conv_set_overrides), copied under a
// lock; every field -1 keeps the library's own choice.
struct Overrides {
    int tile_n, k_bytes, stages, group_m, splits, pair, msub, slices, epilogue, hw_major,
        two_phase, repack, dy_in_place, pdl, weight_groups, ncdhw_in_place, pack_lanes, log;
};
Overrides overrides();

// Record a failure description for conv_last_error() on the calling thread.
void set_last_error(const char* msg);

}  // namespace c3d
