// C ABI of the LLM.int8() decomposed matmul (declarations and contracts in
// include/llmint8.h).  Host side: argument checks, workspace layout, tensor-map
// encoding and kernel launches.  Every step of the path runs in the kernels of
// this library; there is no host or library fallback.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "llmint8.h"
#include "common.cuh"
#include "xpass.cuh"
#include "wquant.cuh"
#include "gemv.cuh"
#include "gemm_tc.cuh"
#include "chain.cuh"

using namespace llmint8;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool probed = false;
    bool supported = false;
    int sms = 0;
    // kernel attributes set on this device, per element format (0 fp16, 1 bf16)
    bool gemm_attr_set[2] = {false, false};
    bool gemv_attr_set[2] = {false, false};
    bool rowq_cluster_attr_set[2] = {false, false};
    bool chain_attr_set = false;
    bool widen_attr_set = false;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

llmint8_status current_device(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LLMINT8_ECUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.probed) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return LLMINT8_ECUDA;
        d.supported = (major == 10 && minor == 3);
        d.sms = sms;
        d.probed = true;
    }
    if (!d.supported) return LLMINT8_EUNSUPPORTED;
    *out = &d;
    return LLMINT8_OK;
}

llmint8_status get_encoder() {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_encode) return LLMINT8_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return LLMINT8_ECUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return LLMINT8_OK;
}

// 2D fp16 tensor [rows, cols] row-major with row pitch `pitch` elements; box
// of box_rows x 64 columns, 128-byte swizzle (the MMA operand layout).
llmint8_status encode_fp16_2d(CUtensorMap* map, const void* base, int rows, int cols, int pitch, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)pitch * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? LLMINT8_OK : LLMINT8_ECUDA;
}

// The GEMM output [rows, cols] row-major with elements of `esize` bytes (2: Y,
// 4: C) for TMA stores: box of 32 rows x 128 bytes, 128-byte swizzle.
llmint8_status encode_out_2d(CUtensorMap* map, void* base, int rows, int cols, int esize) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * esize};
    cuuint32_t box[2] = {(cuuint32_t)(128 / esize), 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_INT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, base,
                          dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? LLMINT8_OK : LLMINT8_ECUDA;
}

// 2D int8 tensor [rows, cols] row-major (pitch = cols bytes); box of box_rows x
// box_cols bytes, no swizzle (rows land box_cols bytes apart in shared memory).
llmint8_status encode_u8_2d(CUtensorMap* map, const void* base, int rows, int cols, int box_rows, int box_cols) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? LLMINT8_OK : LLMINT8_ECUDA;
}

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Layout {
    size_t hdr, bitmap, idx, row_scale, codes, xo, w16o, wq16, total;
    int kp;  // padded pitch of the gathered outlier operands (multiple of 64)
    bool decode;
};

Layout make_layout(int M, int K, int N) {
    Layout L;
    L.decode = M <= LLMINT8_DECODE_MAX_M;
    L.kp = (int)align_up((size_t)K, 64);
    size_t off = 0;
    L.hdr = off;
    off += 256;
    L.bitmap = off;
    off = align_up(off + (size_t)((K + 31) / 32) * 4, 256);
    L.idx = off;
    off = align_up(off + (size_t)K * 4, 256);
    L.row_scale = off;
    off = align_up(off + (size_t)M * 4, 256);
    L.codes = off;
    off = align_up(off + (size_t)M * K * 2, 256);
    L.xo = off;
    off = align_up(off + (size_t)M * L.kp * 2, 256);
    L.w16o = off;
    if (!L.decode) off = align_up(off + (size_t)N * L.kp * 2, 256);
    // prefill: the weight codes as fp16 integers, [N, K] (the GEMM's B operand)
    L.wq16 = align_up(off, 1024);
    if (!L.decode) off = L.wq16 + (size_t)N * K * 2;
    L.total = off;
    return L;
}

bool sizes_ok(int M, int K, int N) { return M >= 1 && K >= 1 && N >= 1 && K <= kMaxK && N <= (1 << 30); }

llmint8_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? LLMINT8_OK : LLMINT8_ECUDA;
}

// Launch with the programmatic stream-serialization attribute when `pdl`: the
// kernel may start while its predecessor in the stream is still running and
// synchronizes with it through griddepcontrol.wait (pdl_wait in the kernels).
template <typename... KArgs, typename... Args>
llmint8_status launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                      Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...) == cudaSuccess ? LLMINT8_OK : LLMINT8_ECUDA;
}

int row_quant_vpt(int K) {
    const int nvec = K / 8;
    if (nvec <= kRowThreads) return 1;
    if (nvec <= 2 * kRowThreads) return 2;
    if (nvec <= 4 * kRowThreads) return 4;
    if (nvec <= 8 * kRowThreads) return 8;
    return 0;
}

// Decode X pass in one clustered row-quantization launch: M <= 16, a finite
// threshold and rows of at most 4096 columns (two 16-byte vectors per thread).
bool cluster_flags_apply(int M, int K, float threshold) {
    const bool use_outliers = !(std::isinf(threshold) && threshold > 0);
    const int vpt = row_quant_vpt(K);
    return M <= LLMINT8_DECODE_MAX_M && use_outliers && (vpt == 1 || vpt == 2);
}

// As launch(), as one thread-block cluster of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
llmint8_status launch_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                              unsigned cluster_x, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster_x;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...) == cudaSuccess ? LLMINT8_OK : LLMINT8_ECUDA;
}


// Checks shared by every entry point that runs part of the matmul.
llmint8_status check_common(const void* X, int M, int K, int N, float threshold, void* workspace, size_t ws_bytes,
                            Layout* L, DeviceInfo** dev) {
    if (!X) return LLMINT8_EINVAL;
    if (!sizes_ok(M, K, N) || std::isnan(threshold)) return LLMINT8_EINVAL;
    if ((K % 16) || (N % 16)) return LLMINT8_EALIGN;
    if (!aligned16(X) || !aligned16(workspace)) return LLMINT8_EALIGN;
    *L = make_layout(M, K, N);
    if (!workspace || ws_bytes < L->total) return LLMINT8_EWORKSPACE;
    return LLMINT8_OK;
}

// Where the outlier slice (A4) reads the rows of W: the full fp16 copy W16, or
// (w8) kept rows W16c through row_map and the dequantized codes for the rest.
struct W16Src {
    bool w8 = false;
    const __half* W16c = nullptr;
    const int32_t* row_map = nullptr;
    int rows = 0;
};

// Checks of the GEMM operands.
llmint8_status check_operands(int M, float threshold, const int8_t* Wq, const float* colScaleW, const void* W16,
                              const void* out, bool write_i32, const W16Src& src = W16Src()) {
    const bool use_outliers = !(std::isinf(threshold) && threshold > 0);
    (void)M;
    if (!Wq || !colScaleW || !out) return LLMINT8_EINVAL;
    if (use_outliers && !W16 && !write_i32 && !src.w8) return LLMINT8_EINVAL;
    if (src.w8 && (src.rows < 0 || (src.rows > 0 && (!src.W16c || !src.row_map)))) return LLMINT8_EINVAL;
    if (src.w8 && src.W16c && !aligned16(src.W16c)) return LLMINT8_EALIGN;
    if (!aligned16(Wq) || !aligned16(colScaleW) || !aligned16(out) || (W16 && !aligned16(W16)))
        return LLMINT8_EALIGN;
    return LLMINT8_OK;
}

struct WsView {
    WsHeader* hdr;
    uint32_t* bitmap;
    int32_t* idx;
    float* row_scale;
    __half* codes;
    __half* xo;
    __half* w16o;
    __half* wq16;
    WsView(void* workspace, const Layout& L) {
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        hdr = reinterpret_cast<WsHeader*>(ws + L.hdr);
        bitmap = reinterpret_cast<uint32_t*>(ws + L.bitmap);
        idx = reinterpret_cast<int32_t*>(ws + L.idx);
        row_scale = reinterpret_cast<float*>(ws + L.row_scale);
        codes = reinterpret_cast<__half*>(ws + L.codes);
        xo = reinterpret_cast<__half*>(ws + L.xo);
        w16o = reinterpret_cast<__half*>(ws + L.w16o);
        wq16 = reinterpret_cast<__half*>(ws + L.wq16);
    }
};

// Prefill rows of at most 4096 columns run k_row_quant_warp, which can also
// write the gathered outlier rows of W16 for the GEMM (no separate gather).
// Only while its M/8 CTAs are enough for the N/16 column groups (at most 8
// groups each): at M = 32, N = 11008 the 4 CTAs took 147 us for 688 groups,
// where the separate gather kernel runs N/64 CTAs.
bool rowq_gathers_w16(bool decode, int M, int K, int N, float threshold, bool write_i32, const void* W16) {
    const bool use_outliers = !(std::isinf(threshold) && threshold > 0);
    const bool enough_ctas = (size_t)((M + kRowsPerCta - 1) / kRowsPerCta) * 8 >= (size_t)(N / kGatherCols);
    return !decode && K <= 4096 && enough_ctas && use_outliers && !write_i32 && W16 != nullptr;
}

// Caller-owned destinations of A2 (llmint8_quantize_x): int8 codes [M, K] and
// row scales [M] in place of the workspace fields; no gathered outlier values.
struct XpassOut {
    int8_t* codes = nullptr;
    float* row_scale = nullptr;
};

// A1 + A2 into the workspace; with gather_w16 also the A4 operand W16oT.
template <typename T>
llmint8_status xpass_launch(const void* X, int M, int K, float threshold, void* workspace, const Layout& L,
                            DeviceInfo* dev, cudaStream_t s, const void* W16 = nullptr, int N = 0,
                            bool gather_w16 = false, const XpassOut& dst = XpassOut()) {
    const bool use_outliers = !(std::isinf(threshold) && threshold > 0);
    const WsView w(workspace, L);
    const __half* Xh = static_cast<const __half*>(X);
    llmint8_status st;

    // A1: outlier columns.  With one row group (always for M <= 64) each scan CTA
    // stores its bitmap words directly and CTA 0 resets the error word; with
    // several row groups the words are OR-ed atomically into a zeroed map.
    // Short decode rows: the row-quantization CTAs form one cluster and find the
    // outlier columns themselves (no scan kernel).  Longer rows keep the scan:
    // its K / 256 CTAs share the flag work that one CTA per row would do alone.
    const bool cluster = cluster_flags_apply(M, K, threshold);
    const int gx = (K + kScanCols - 1) / kScanCols;
    int gy = 1;
    if (M > 64) {
        gy = (M + 7) / 8;
        const int cap = (dev->sms * 8 + gx - 1) / gx;
        if (gy > cap) gy = cap;
        if (gy < 1) gy = 1;
    }
    if (use_outliers && !cluster) {
        if (gy > 1 && cudaMemsetAsync(static_cast<uint8_t*>(workspace) + L.hdr, 0, L.idx - L.hdr, s) != cudaSuccess)
            return LLMINT8_ECUDA;
        st = launch(k_outlier_scan<T>, dim3(gx, gy), dim3(kScanThreads), 0, s, true, Xh, M, K, threshold, w.bitmap,
                    gy > 1 ? nullptr : w.hdr);
        if (st != LLMINT8_OK) return st;
    }

    // A2: row scales and codes (+ the gathered outlier columns of X)
    RowQuantArgs ra{};
    ra.X = Xh;
    ra.M = M;
    ra.K = K;
    ra.bitmap = w.bitmap;
    ra.hdr = w.hdr;
    ra.outlier_idx = w.idx;
    ra.row_scale = dst.codes ? dst.row_scale : w.row_scale;
    ra.codes = dst.codes ? static_cast<void*>(dst.codes) : static_cast<void*>(w.codes);
    // int8 for the decode GEMV (and caller buffers), fp16 values for the tensor-core GEMM
    ra.codes_fp16 = (L.decode || dst.codes) ? 0 : 1;
    ra.xo = (use_outliers && !dst.codes) ? w.xo : nullptr;
    ra.xo_pitch = L.kp;
    ra.no_outliers = use_outliers ? 0 : 1;
    ra.clear_status = (use_outliers && !cluster) ? 0 : 1;
    ra.t = threshold;
    ra.cluster_flags = cluster ? 1 : 0;
    const bool pdl = true;
    if (cluster) {
        {
            std::lock_guard<std::mutex> lock(g_mu);
            if (!dev->rowq_cluster_attr_set[Fmt<T>::kBF16]) {  // clusters of up to 16 CTAs (M <= 16)
                if (cudaFuncSetAttribute(k_row_quant<1, T>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                        cudaSuccess ||
                    cudaFuncSetAttribute(k_row_quant<2, T>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                        cudaSuccess)
                    return LLMINT8_ECUDA;
                dev->rowq_cluster_attr_set[Fmt<T>::kBF16] = true;
            }
        }
        const unsigned cm = (unsigned)M;
        return row_quant_vpt(K) == 1 ? launch_cluster(k_row_quant<1, T>, dim3(M), dim3(kRowThreads), 0, s, pdl, cm, ra)
                                     : launch_cluster(k_row_quant<2, T>, dim3(M), dim3(kRowThreads), 0, s, pdl, cm, ra);
    }
    if (dst.codes) gather_w16 = false;
    ra.W16 = gather_w16 ? static_cast<const __half*>(W16) : nullptr;
    ra.N = N;
    ra.w16o = gather_w16 ? w.w16o : nullptr;
    ra.w16o_pitch = L.kp;
    if (!L.decode && K <= 4096) {  // many short rows: one warp per row
        // rows per CTA: as many as spread the rows over two CTAs per SM, at most 8
        const int per_cta = std::max(1, std::min(kRowsPerCta, (M + 2 * dev->sms - 1) / (2 * dev->sms)));
        ra.rows_per_cta = per_cta;
        const dim3 grid((M + per_cta - 1) / per_cta), block(kRowsPerCta * 32);
        if (K <= 1024) return launch(k_row_quant_warp<4, T>, grid, block, 0, s, pdl, ra);
        if (K <= 2048) return launch(k_row_quant_warp<8, T>, grid, block, 0, s, pdl, ra);
        return launch(k_row_quant_warp<16, T>, grid, block, 0, s, pdl, ra);
    }
    switch (row_quant_vpt(K)) {
        case 1: return launch(k_row_quant<1, T>, dim3(M), dim3(kRowThreads), 0, s, pdl, ra);
        case 2: return launch(k_row_quant<2, T>, dim3(M), dim3(kRowThreads), 0, s, pdl, ra);
        case 4: return launch(k_row_quant<4, T>, dim3(M), dim3(kRowThreads), 0, s, pdl, ra);
        case 8: return launch(k_row_quant<8, T>, dim3(M), dim3(kRowThreads), 0, s, pdl, ra);
        default: return launch(k_row_quant<0, T>, dim3(M), dim3(kRowThreads), 0, s, pdl, ra);
    }
}

// Tile shape and grid of the prefill GEMM (persistent over ctas_or_clusters).
struct GemmPlan {
    bool pair;
    int bn, ctas_or_clusters;
};

GemmPlan gemm_plan(int M, int N, int K, int sms) {
    GemmPlan g;
    g.pair = M > kBM && sms >= 2;
    const int tiles_m = g.pair ? (M + 2 * kBM - 1) / (2 * kBM) : (M + kBM - 1) / kBM;
    const int slots = g.pair ? sms / 2 : sms;
    if (g.pair)
        g.bn = tiles_m * ((N + kBN - 1) / kBN) * 10 < 6 * slots ? 128 : kBN;
    else
        g.bn = tiles_m * ((N + kBN - 1) / kBN) * 2 <= slots ? 128 : kBN;
    const int tiles = tiles_m * ((N + g.bn - 1) / g.bn);
    g.ctas_or_clusters = tiles < slots ? tiles : slots;
    (void)K;
    return g;
}

// k_widen_codes over nbytes int8 codes (-> exact fp16 integers at dst).
llmint8_status widen_launch(const int8_t* src, __half* dst, size_t nbytes, bool src_constant, WsHeader* err,
                            DeviceInfo* dev, cudaStream_t s, bool pdl) {
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!dev->widen_attr_set) {
            if (cudaFuncSetAttribute(k_widen_codes, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWidenSmem) !=
                cudaSuccess)
                return LLMINT8_ECUDA;
            dev->widen_attr_set = true;
        }
    }
    const size_t nchunks = (nbytes + kWidenChunk - 1) / kWidenChunk;
    const unsigned grid = (unsigned)(nchunks < (size_t)dev->sms ? nchunks : (size_t)dev->sms);
    return launch(k_widen_codes, dim3(grid), dim3(kWidenThreads), kWidenSmem, s, pdl, src, dst, nbytes,
                  src_constant ? 1 : 0, err, kDefaultSpinLimit);
}

// A3 + A4 + A5 from the workspace an xpass_launch of the same problem filled.
template <typename T>
llmint8_status gemm_launch(const void* X, int M, int K, int N, float threshold, const int8_t* Wq,
                           const float* colScaleW, const void* W16, void* out, bool write_i32,
                           void* workspace, const Layout& L, DeviceInfo* dev, cudaStream_t s,
                           bool w16o_ready = false, const W16Src& src = W16Src(),
                           const int8_t* codes8 = nullptr) {
    const bool use_outliers = !(std::isinf(threshold) && threshold > 0);
    const WsView w(workspace, L);
    llmint8_status st;

    if (L.decode) {
        GemvArgs ga;
        // the X pass's int8 codes, or the caller's (llmint8_gemm_i32)
        ga.codes = codes8 ? codes8 : reinterpret_cast<const int8_t*>(w.codes);
        ga.Wq = Wq;
        ga.col_scale = colScaleW;
        ga.row_scale = w.row_scale;
        ga.W16 = static_cast<const __half*>(W16);
        ga.hdr = w.hdr;
        ga.outlier_idx = w.idx;
        ga.xo = w.xo;
        ga.xo_pitch = L.kp;
        ga.out = out;
        ga.M = M;
        ga.K = K;
        ga.N = N;
        const int ksteps = (K + 63) / 64;
        ga.k_per_warp = ((ksteps + kGemvWarps - 1) / kGemvWarps) * 64;
        ga.use_outliers = use_outliers ? 1 : 0;
        ga.w8 = src.w8 ? 1 : 0;
        ga.W16c = src.W16c;
        ga.row_map = src.row_map;
        ga.w16_rows = src.rows;
        {
            std::lock_guard<std::mutex> lock(g_mu);
            if (!dev->gemv_attr_set[Fmt<T>::kBF16]) {
                const int m8 = (int)gemv_dyn_smem(8), m16 = (int)gemv_dyn_smem(16);
                if (cudaFuncSetAttribute(k_gemv_decode<1, true, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, m8) !=
                        cudaSuccess ||
                    cudaFuncSetAttribute(k_gemv_decode<1, false, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, m8) !=
                        cudaSuccess ||
                    cudaFuncSetAttribute(k_gemv_decode<2, true, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, m16) !=
                        cudaSuccess ||
                    cudaFuncSetAttribute(k_gemv_decode<2, false, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, m16) !=
                        cudaSuccess ||
                    cudaFuncSetAttribute(k_gemv_decode_tiles<1, true, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         m8) != cudaSuccess ||
                    cudaFuncSetAttribute(k_gemv_decode_tiles<1, false, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         m8) != cudaSuccess)
                    return LLMINT8_ECUDA;
                dev->gemv_attr_set[Fmt<T>::kBF16] = true;
            }
        }
        const dim3 block(kGemvWarps * 32);
        const int ntiles = N / kGemvCols, slots = 2 * dev->sms;  // two CTAs per SM
        if (M <= 8) {
            if (ntiles > slots) {  // one-tile CTAs would need several waves: persistent grid
                const dim3 grid(slots);
                return write_i32 ? launch(k_gemv_decode_tiles<1, true, T>, grid, block, gemv_dyn_smem(M), s, true, ga)
                                 : launch(k_gemv_decode_tiles<1, false, T>, grid, block, gemv_dyn_smem(M), s, true, ga);
            }
            const dim3 grid(ntiles);
            return write_i32 ? launch(k_gemv_decode<1, true, T>, grid, block, gemv_dyn_smem(M), s, true, ga)
                             : launch(k_gemv_decode<1, false, T>, grid, block, gemv_dyn_smem(M), s, true, ga);
        }
        // up to 16 rows: the persistent form measured slower (its per-tile
        // epilogue costs more than the waves it removes), one-tile CTAs
        const dim3 grid(ntiles);
        return write_i32 ? launch(k_gemv_decode<2, true, T>, grid, block, gemv_dyn_smem(M), s, true, ga)
                         : launch(k_gemv_decode<2, false, T>, grid, block, gemv_dyn_smem(M), s, true, ga);
    }

    // A4 operand: gathered, transposed outlier rows of W16 (unless the X pass wrote it)
    if (use_outliers && !write_i32 && !w16o_ready) {
        const W8Rows w8{src.W16c, src.row_map, src.rows, Wq, K, colScaleW};
        st = launch(k_gather_w16_outlier_rows<T>, dim3((N + 63) / 64), dim3(256), 0, s, true,
                    src.w8 ? nullptr : static_cast<const __half*>(W16), N, (const WsHeader*)w.hdr,
                    (const int32_t*)w.idx, w.w16o, L.kp, w8);
        if (st != LLMINT8_OK) return st;
    }
    // Tiling.  CTA pairs (256 x 256 tiles, each CTA loading 128 columns of B)
    // once M spans two 128-row tiles; 256 x 128 pair tiles when the wide ones
    // would give fewer clusters than 60 % of the cluster slots (medium M); one
    // CTA per 128 x 256 tile below, or 128 x 128 when that still leaves half the
    // SMs idle.
    const GemmPlan g = gemm_plan(M, N, K, dev->sms);
    const int b_rows = g.pair ? g.bn / 2 : g.bn;
    // A3 operand: the int8 codes widened to exact fp16 integers in the scratch
    if ((st = widen_launch(Wq, w.wq16, (size_t)N * K, true, w.hdr, dev, s, true)) != LLMINT8_OK) return st;
    if ((st = get_encoder()) != LLMINT8_OK) return st;
    CUtensorMap tm_a, tm_b, tm_xo, tm_wo, tm_out;
    if ((st = encode_fp16_2d(&tm_a, w.codes, M, K, K, kBM)) != LLMINT8_OK) return st;
    if ((st = encode_fp16_2d(&tm_b, w.wq16, N, K, K, b_rows)) != LLMINT8_OK) return st;
    if ((st = encode_fp16_2d(&tm_xo, w.xo, M, L.kp, L.kp, kBM)) != LLMINT8_OK) return st;
    if ((st = encode_fp16_2d(&tm_wo, w.w16o, N, L.kp, L.kp, b_rows)) != LLMINT8_OK) return st;
    if ((st = encode_out_2d(&tm_out, out, M, N, write_i32 ? 4 : 2)) != LLMINT8_OK) return st;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!dev->gemm_attr_set[Fmt<T>::kBF16]) {
            const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
            if (cudaFuncSetAttribute(k_gemm_tc<false, false, T, 256>, attr, (int)kGemmSmem) != cudaSuccess ||
                cudaFuncSetAttribute(k_gemm_tc<true, false, T, 256>, attr, (int)kGemmSmem) != cudaSuccess ||
                cudaFuncSetAttribute(k_gemm_tc<false, false, T, 128>, attr, (int)kGemmSmem) != cudaSuccess ||
                cudaFuncSetAttribute(k_gemm_tc<true, false, T, 128>, attr, (int)kGemmSmem) != cudaSuccess ||
                cudaFuncSetAttribute(k_gemm_tc<false, true, T, 256>, attr, (int)kGemmSmem) != cudaSuccess ||
                cudaFuncSetAttribute(k_gemm_tc<true, true, T, 256>, attr, (int)kGemmSmem) != cudaSuccess ||
                cudaFuncSetAttribute(k_gemm_tc<false, true, T, 128>, attr, (int)kGemmSmem) != cudaSuccess ||
                cudaFuncSetAttribute(k_gemm_tc<true, true, T, 128>, attr, (int)kGemmSmem) != cudaSuccess)
                return LLMINT8_ECUDA;
            dev->gemm_attr_set[Fmt<T>::kBF16] = true;
        }
    }
    GemmArgs ga;
    ga.row_scale = w.row_scale;
    ga.col_scale = colScaleW;
    ga.hdr = w.hdr;
    ga.err = w.hdr;
    ga.M = M;
    ga.N = N;
    ga.K = K;
    // the int32 accumulator leaves the outlier slice out (it is not part of C)
    ga.use_outliers = (use_outliers && !write_i32) ? 1 : 0;
    ga.spin_limit = kDefaultSpinLimit;
    const dim3 block(kGemmThreads);
    if (g.pair) {
        const dim3 grid(2 * g.ctas_or_clusters);
        if (g.bn == 128)
            return write_i32 ? launch_cluster(k_gemm_tc<true, true, T, 128>, grid, block, kGemmSmem, s, true, 2u, tm_a,
                                              tm_b, tm_xo, tm_wo, tm_out, ga)
                             : launch_cluster(k_gemm_tc<false, true, T, 128>, grid, block, kGemmSmem, s, true, 2u,
                                              tm_a, tm_b, tm_xo, tm_wo, tm_out, ga);
        return write_i32 ? launch_cluster(k_gemm_tc<true, true, T, 256>, grid, block, kGemmSmem, s, true, 2u, tm_a,
                                          tm_b, tm_xo, tm_wo, tm_out, ga)
                         : launch_cluster(k_gemm_tc<false, true, T, 256>, grid, block, kGemmSmem, s, true, 2u, tm_a,
                                          tm_b, tm_xo, tm_wo, tm_out, ga);
    }
    const dim3 grid(g.ctas_or_clusters);
    if (g.bn == 128)
        return write_i32 ? launch(k_gemm_tc<true, false, T, 128>, grid, block, kGemmSmem, s, true, tm_a, tm_b, tm_xo,
                                  tm_wo, tm_out, ga)
                         : launch(k_gemm_tc<false, false, T, 128>, grid, block, kGemmSmem, s, true, tm_a, tm_b, tm_xo,
                                  tm_wo, tm_out, ga);
    return write_i32 ? launch(k_gemm_tc<true, false, T, 256>, grid, block, kGemmSmem, s, true, tm_a, tm_b, tm_xo,
                              tm_wo, tm_out, ga)
                     : launch(k_gemm_tc<false, false, T, 256>, grid, block, kGemmSmem, s, true, tm_a, tm_b, tm_xo,
                              tm_wo, tm_out, ga);
}

// Kernels one matmul call launches (the plan matmul_impl follows).
int kernels_per_call(int M, int K, int N, float threshold, bool write_i32) {
    const bool use_outliers = !(std::isinf(threshold) && threshold > 0);
    // short decode rows find their outlier columns in the row-quantization
    // cluster: no scan kernel
    const bool scan = use_outliers && !cluster_flags_apply(M, K, threshold);
    int n = (scan ? 1 : 0) + 1 + 1;  // scan, row quant, GEMV / GEMM
    // outlier rows of W16 for the GEMM, unless the row quantization gathers them
    if (M > LLMINT8_DECODE_MAX_M && use_outliers && !write_i32 &&
        !rowq_gathers_w16(false, M, K, N, threshold, write_i32, reinterpret_cast<const void*>(1)))
        n += 1;
    // the codes widened to fp16 for the tensor cores
    if (M > LLMINT8_DECODE_MAX_M) n += 1;
    return n;
}

llmint8_status matmul_impl(const void* X, int M, int K, int N, float threshold, const int8_t* Wq,
                           const float* colScaleW, const void* W16, void* out, bool write_i32,
                           void* workspace, size_t ws_bytes, void* stream, const W16Src& src = W16Src(),
                           bool bf16 = false) {
    Layout L;
    DeviceInfo* dev = nullptr;
    llmint8_status st = check_common(X, M, K, N, threshold, workspace, ws_bytes, &L, &dev);
    if (st != LLMINT8_OK) return st;
    if ((st = check_operands(M, threshold, Wq, colScaleW, W16, out, write_i32, src)) != LLMINT8_OK) return st;
    if ((st = current_device(&dev)) != LLMINT8_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the row quantization gathers only from a full fp16 copy (W16 is null in w8 mode)
    const bool gw = !src.w8 && rowq_gathers_w16(L.decode, M, K, N, threshold, write_i32, W16);
    const void* W16g = src.w8 ? nullptr : W16;
    if (bf16) {
        if ((st = xpass_launch<__nv_bfloat16>(X, M, K, threshold, workspace, L, dev, s, W16, N, gw)) != LLMINT8_OK)
            return st;
        return gemm_launch<__nv_bfloat16>(X, M, K, N, threshold, Wq, colScaleW, W16g, out, write_i32,
                                          workspace, L, dev, s, gw, src);
    }
    if ((st = xpass_launch<__half>(X, M, K, threshold, workspace, L, dev, s, W16, N, gw)) != LLMINT8_OK) return st;
    return gemm_launch<__half>(X, M, K, N, threshold, Wq, colScaleW, W16g, out, write_i32, workspace, L, dev,
                               s, gw, src);
}

// ---- decode chain (chain.cuh): the streaming GEMV for up to 4 rows of X ----
constexpr size_t kMaxDynSmem = 232448;  // 227 KB, the opt-in limit of one CTA
constexpr size_t kSmemPerSM = 233472;   // 228 KB, of which 1 KB per resident CTA is reserved

// the kernel's static shared memory (under 1 KB) counts against the same limit
constexpr size_t kChainMaxDynSmem = kMaxDynSmem - 1024;

bool chain_shape_ok(int M, int K) {
    return M >= 1 && M <= kChainMaxM && K >= kChainStageK && chain_smem(M, K) <= kChainMaxDynSmem;
}

template <int MR>
bool set_chain_attrs() {
    const int m = (int)kChainMaxDynSmem;
    const auto a = cudaFuncAttributeMaxDynamicSharedMemorySize;
    return cudaFuncSetAttribute(k_gemv_chain<MR, false, false>, a, m) == cudaSuccess &&
           cudaFuncSetAttribute(k_gemv_chain<MR, false, true>, a, m) == cudaSuccess &&
           cudaFuncSetAttribute(k_gemv_chain<MR, true, false>, a, m) == cudaSuccess &&
           cudaFuncSetAttribute(k_gemv_chain<MR, true, true>, a, m) == cudaSuccess;
}

template <int MR>
llmint8_status chain_launch_m(const CUtensorMap& tw, const GemvArgs& ga, const ChainArgs& ch, dim3 grid,
                              size_t smem, cudaStream_t s) {
    const dim3 block(kChainThreads);
    if (ch.in != nullptr)
        return ch.out != nullptr ? launch(k_gemv_chain<MR, true, true>, grid, block, smem, s, true, tw, ga, ch)
                                 : launch(k_gemv_chain<MR, true, false>, grid, block, smem, s, true, tw, ga, ch);
    return ch.out != nullptr ? launch(k_gemv_chain<MR, false, true>, grid, block, smem, s, true, tw, ga, ch)
                             : launch(k_gemv_chain<MR, false, false>, grid, block, smem, s, true, tw, ga, ch);
}

// One launch of k_gemv_chain: a persistent grid of up to two CTAs per SM.
llmint8_status chain_launch(const GemvArgs& ga, const ChainArgs& ch, DeviceInfo* dev, cudaStream_t s) {
    llmint8_status st;
    if ((st = get_encoder()) != LLMINT8_OK) return st;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!dev->chain_attr_set) {
            if (!set_chain_attrs<1>() || !set_chain_attrs<2>() || !set_chain_attrs<3>() || !set_chain_attrs<4>())
                return LLMINT8_ECUDA;
            dev->chain_attr_set = true;
        }
    }
    CUtensorMap tw;
    if ((st = encode_u8_2d(&tw, ga.Wq, ga.N, ga.K, kChainCols, kChainBoxK)) != LLMINT8_OK) return st;
    const size_t smem = chain_smem(ga.M, ga.K);
    const int per_sm = 2 * (smem + 1024) <= kSmemPerSM ? 2 : 1;
    const int strips = ga.N / kChainCols;
    const dim3 grid(strips < per_sm * dev->sms ? strips : per_sm * dev->sms);
    switch (ga.M) {
        case 1: return chain_launch_m<1>(tw, ga, ch, grid, smem, s);
        case 2: return chain_launch_m<2>(tw, ga, ch, grid, smem, s);
        case 3: return chain_launch_m<3>(tw, ga, ch, grid, smem, s);
        default: return chain_launch_m<4>(tw, ga, ch, grid, smem, s);
    }
}

// Waits on a barrier nothing completes, bounded by spin_limit polls, then
// records the timeout in the error word.
__global__ void k_selftest_timeout(WsHeader* hdr, uint32_t spin_limit) {
    __shared__ uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!mbar_wait_bounded(&bar, 0, spin_limit, &abort_flag)) record_error(hdr, kStatusTimeout, 99);
    }
}

}  // namespace

// A0 for W of element format T (fp16 or bf16)
template <typename T>
llmint8_status quantize_weight_impl(const void* W, int K, int N, int8_t* Wq, float* colScaleW, void* stream) {
    if (!W || !Wq || !colScaleW) return LLMINT8_EINVAL;
    if (K < 1 || N < 1 || K > (1 << 30) || N > (1 << 30)) return LLMINT8_EINVAL;
    if ((K % 16) || (N % 16)) return LLMINT8_EALIGN;
    if (!aligned16(W) || !aligned16(Wq) || !aligned16(colScaleW)) return LLMINT8_EALIGN;
    DeviceInfo* dev = nullptr;
    llmint8_status st = current_device(&dev);
    if (st != LLMINT8_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(colScaleW, 0, (size_t)N * 4, s) != cudaSuccess) return LLMINT8_ECUDA;
    const int gx = (N + 255) / 256;
    int gy = (K + 7) / 8;
    const int cap = (dev->sms * 8 + gx - 1) / gx;
    if (gy > cap) gy = cap;
    if (gy < 1) gy = 1;
    k_col_absmax<T><<<dim3(gx, gy), 256, 0, s>>>(static_cast<const __half*>(W), K, N, colScaleW);
    if ((st = launch_status()) != LLMINT8_OK) return st;
    k_quantize_weight_tile<T><<<dim3((N + 63) / 64, (K + 63) / 64), 256, 0, s>>>(
        static_cast<const __half*>(W), K, N, colScaleW, Wq);
    return launch_status();
}

extern "C" {

const char* llmint8_status_str(int status) {
    switch (status) {
        case LLMINT8_OK: return "LLMINT8_OK";
        case LLMINT8_EINVAL: return "LLMINT8_EINVAL: invalid argument";
        case LLMINT8_EALIGN: return "LLMINT8_EALIGN: K/N not a multiple of 16 or pointer not 16-byte aligned";
        case LLMINT8_EWORKSPACE: return "LLMINT8_EWORKSPACE: workspace missing or too small";
        case LLMINT8_ECUDA: return "LLMINT8_ECUDA: CUDA runtime call or kernel launch failed";
        case LLMINT8_ETIMEOUT: return "LLMINT8_ETIMEOUT: a bounded device wait gave up";
        case LLMINT8_EUNSUPPORTED: return "LLMINT8_EUNSUPPORTED: device is not sm_103";
        default: return "LLMINT8: unknown status";
    }
}

llmint8_status llmint8_quantize_weight(const void* W, int K, int N, int8_t* Wq, float* colScaleW, void* stream) {
    return quantize_weight_impl<__half>(W, K, N, Wq, colScaleW, stream);
}

llmint8_status llmint8_quantize_weight_bf16(const void* W, int K, int N, int8_t* Wq, float* colScaleW, void* stream) {
    return quantize_weight_impl<__nv_bfloat16>(W, K, N, Wq, colScaleW, stream);
}

llmint8_status llmint8_matmul_bf16(const void* X, int M, int K, int N, float threshold, const int8_t* Wq,
                                   const float* colScaleW, const void* W16, void* Y, void* workspace,
                                   size_t workspace_bytes, void* stream) {
    return matmul_impl(X, M, K, N, threshold, Wq, colScaleW, W16, Y, false, workspace, workspace_bytes,
                       stream, W16Src(), true);
}

llmint8_status llmint8_matmul_i32_bf16(const void* X, int M, int K, int N, float threshold, const int8_t* Wq,
                                       const float* colScaleW, int32_t* C, void* workspace,
                                       size_t workspace_bytes, void* stream) {
    return matmul_impl(X, M, K, N, threshold, Wq, colScaleW, nullptr, C, true, workspace, workspace_bytes,
                       stream, W16Src(), true);
}

size_t llmint8_workspace_bytes(int M, int K, int N) {
    if (!sizes_ok(M, K, N)) return 0;
    return make_layout(M, K, N).total;
}

llmint8_status llmint8_matmul(const void* X, int M, int K, int N, float threshold, const int8_t* Wq,
                              const float* colScaleW, const void* W16, void* Y, void* workspace,
                              size_t workspace_bytes, void* stream) {
    return matmul_impl(X, M, K, N, threshold, Wq, colScaleW, W16, Y, false, workspace, workspace_bytes,
                       stream);
}

llmint8_status llmint8_matmul_host(const void* X_host, void* X, int M, int K, int N, float threshold,
                                   const int8_t* Wq, const float* colScaleW, const void* W16, void* Y,
                                   void* Y_host, void* workspace, size_t workspace_bytes, void* stream) {
    if (!X_host || !Y_host || !Y) return LLMINT8_EINVAL;
    // every argument of the device call is checked before the first copy is enqueued
    Layout L;
    DeviceInfo* dev = nullptr;
    llmint8_status st = check_common(X, M, K, N, threshold, workspace, workspace_bytes, &L, &dev);
    if (st != LLMINT8_OK) return st;
    if ((st = check_operands(M, threshold, Wq, colScaleW, W16, Y, false)) != LLMINT8_OK) return st;
    if ((st = current_device(&dev)) != LLMINT8_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(X, X_host, (size_t)M * K * 2, cudaMemcpyHostToDevice, s) != cudaSuccess) return LLMINT8_ECUDA;
    if ((st = llmint8_matmul(X, M, K, N, threshold, Wq, colScaleW, W16, Y, workspace, workspace_bytes, stream)) !=
        LLMINT8_OK)
        return st;
    return cudaMemcpyAsync(Y_host, Y, (size_t)M * N * 2, cudaMemcpyDeviceToHost, s) == cudaSuccess ? LLMINT8_OK
                                                                                                  : LLMINT8_ECUDA;
}

llmint8_status llmint8_matmul_w8(const void* X, int M, int K, int N, float threshold, const int8_t* Wq,
                                 const float* colScaleW, const void* W16c, const int32_t* row_map,
                                 int w16_rows, void* Y, void* workspace, size_t workspace_bytes, void* stream) {
    W16Src src;
    src.w8 = true;
    src.W16c = static_cast<const __half*>(W16c);
    src.row_map = row_map;
    src.rows = w16_rows;
    return matmul_impl(X, M, K, N, threshold, Wq, colScaleW, nullptr, Y, false, workspace, workspace_bytes,
                       stream, src);
}

llmint8_status llmint8_pack_w16_rows(const void* W16, int K, int N, const int32_t* rows, int w16_rows, void* W16c,
                                     int32_t* row_map, void* stream) {
    if (!W16 || !row_map || K <= 0 || N <= 0 || K > kMaxK || w16_rows < 0 ||
        (w16_rows > 0 && (!rows || !W16c)))
        return LLMINT8_EINVAL;
    if ((N % 16) || !aligned16(W16) || (W16c && !aligned16(W16c))) return LLMINT8_EALIGN;
    DeviceInfo* dev = nullptr;
    llmint8_status st = current_device(&dev);
    if (st != LLMINT8_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int gk = (K + 255) / 256;
    if ((st = launch(k_row_map_clear, dim3(gk < 1024 ? gk : 1024), dim3(256), 0, s, false, row_map, K)) != LLMINT8_OK)
        return st;
    if (w16_rows == 0) return LLMINT8_OK;
    const size_t work = (size_t)w16_rows * (N / 8);
    const size_t gp = (work + 255) / 256;
    return launch(k_pack_w16_rows, dim3(gp < 4096 ? (unsigned)gp : 4096u), dim3(256), 0, s, false,
                  static_cast<const __half*>(W16), K, N, rows, w16_rows, static_cast<__half*>(W16c), row_map);
}

llmint8_status llmint8_matmul_int8(const void* X, int M, int K, int N, const int8_t* Wq, const float* colScaleW,
                                   void* Y, void* workspace, size_t workspace_bytes,
                                   void* stream) {
    return matmul_impl(X, M, K, N, INFINITY, Wq, colScaleW, nullptr, Y, false, workspace, workspace_bytes,
                       stream);
}

llmint8_status llmint8_matmul_i32(const void* X, int M, int K, int N, float threshold, const int8_t* Wq,
                                  const float* colScaleW, int32_t* C, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    return matmul_impl(X, M, K, N, threshold, Wq, colScaleW, nullptr, C, true, workspace, workspace_bytes,
                       stream);
}

llmint8_status llmint8_gemm_i32(const int8_t* Xq, const int8_t* Wq, int M, int K, int N, int32_t* C,
                                void* workspace, size_t workspace_bytes, void* stream) {
    if (!Xq || !Wq || !C || !sizes_ok(M, K, N)) return LLMINT8_EINVAL;
    if ((K % 16) || (N % 16)) return LLMINT8_EALIGN;
    if (!aligned16(Xq) || !aligned16(Wq) || !aligned16(C) || !aligned16(workspace)) return LLMINT8_EALIGN;
    const Layout L = make_layout(M, K, N);
    if (!workspace || workspace_bytes < L.total) return LLMINT8_EWORKSPACE;
    DeviceInfo* dev = nullptr;
    llmint8_status st = current_device(&dev);
    if (st != LLMINT8_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (L.decode)  // the GEMV reads the caller's codes where the X pass would leave its own
        return gemm_launch<__half>(nullptr, M, K, N, INFINITY, Wq, nullptr, nullptr, C, true, workspace, L, dev, s,
                                   false, W16Src(), Xq);
    // the tensor-core GEMM reads the codes as exact fp16 integers from the workspace
    const WsView w(workspace, L);
    if ((st = widen_launch(Xq, w.codes, (size_t)M * K, false, w.hdr, dev, s, true)) != LLMINT8_OK) return st;
    return gemm_launch<__half>(nullptr, M, K, N, INFINITY, Wq, nullptr, nullptr, C, true, workspace, L, dev, s);
}

llmint8_status llmint8_xpass(const void* X, int M, int K, int N, float threshold, void* workspace,
                             size_t workspace_bytes, void* stream) {
    Layout L;
    DeviceInfo* dev = nullptr;
    llmint8_status st = check_common(X, M, K, N, threshold, workspace, workspace_bytes, &L, &dev);
    if (st != LLMINT8_OK) return st;
    if ((st = current_device(&dev)) != LLMINT8_OK) return st;
    return xpass_launch<__half>(X, M, K, threshold, workspace, L, dev, static_cast<cudaStream_t>(stream));
}

llmint8_status llmint8_quantize_x(const void* X, int M, int K, float threshold, int8_t* Xq, float* rowScaleX,
                                  void* workspace, size_t workspace_bytes, void* stream) {
    Layout L;
    DeviceInfo* dev = nullptr;
    // the workspace holds the outlier set; its codes field is not used (N = 16
    // keeps the layout at its smallest)
    llmint8_status st = check_common(X, M, K, 16, threshold, workspace, workspace_bytes, &L, &dev);
    if (st != LLMINT8_OK) return st;
    if (!Xq || !rowScaleX) return LLMINT8_EINVAL;
    if (!aligned16(Xq) || !aligned16(rowScaleX)) return LLMINT8_EALIGN;
    if ((st = current_device(&dev)) != LLMINT8_OK) return st;
    XpassOut dst;
    dst.codes = Xq;
    dst.row_scale = rowScaleX;
    return xpass_launch<__half>(X, M, K, threshold, workspace, L, dev, static_cast<cudaStream_t>(stream), nullptr, 0,
                                false, dst);
}

llmint8_status llmint8_read_outliers(const void* workspace, int K, int* count, int32_t* idx_host, int capacity,
                                     void* stream) {
    if (!workspace || !count || K < 1 || K > kMaxK || capacity < 0 || (capacity > 0 && !idx_host))
        return LLMINT8_EINVAL;
    // the header and the outlier list sit at offsets that depend on K only
    const Layout L = make_layout(1, K, 16);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return LLMINT8_ECUDA;
    const uint8_t* ws = static_cast<const uint8_t*>(workspace);
    int32_t n = 0;
    if (cudaMemcpy(&n, ws + L.hdr + offsetof(WsHeader, outlier_count), 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        return LLMINT8_ECUDA;
    if (n < 0 || n > K) return LLMINT8_EINVAL;  // not a workspace an X pass of this K filled
    *count = n;
    const int m = n < capacity ? n : capacity;
    if (m > 0 && cudaMemcpy(idx_host, ws + L.idx, (size_t)m * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        return LLMINT8_ECUDA;
    return LLMINT8_OK;
}

llmint8_status llmint8_gemm(const void* X, int M, int K, int N, float threshold, const int8_t* Wq,
                            const float* colScaleW, const void* W16, void* Y, void* workspace,
                            size_t workspace_bytes, void* stream) {
    Layout L;
    DeviceInfo* dev = nullptr;
    llmint8_status st = check_common(X, M, K, N, threshold, workspace, workspace_bytes, &L, &dev);
    if (st != LLMINT8_OK) return st;
    if ((st = check_operands(M, threshold, Wq, colScaleW, W16, Y, false)) != LLMINT8_OK) return st;
    if ((st = current_device(&dev)) != LLMINT8_OK) return st;
    return gemm_launch<__half>(X, M, K, N, threshold, Wq, colScaleW, W16, Y, false, workspace, L, dev,
                       static_cast<cudaStream_t>(stream));
}

int llmint8_kernels_per_call(int M, int K, int N, float threshold, int write_i32) {
    if (!sizes_ok(M, K, N) || std::isnan(threshold)) return -1;
    return kernels_per_call(M, K, N, threshold, write_i32 != 0);
}

llmint8_status llmint8_workspace_layout(int M, int K, int N, size_t* offsets) {
    if (!offsets || !sizes_ok(M, K, N)) return LLMINT8_EINVAL;
    const Layout L = make_layout(M, K, N);
    offsets[LLMINT8_WS_STATUS] = L.hdr + offsetof(WsHeader, status);
    offsets[LLMINT8_WS_OUTLIER_COUNT] = L.hdr + offsetof(WsHeader, outlier_count);
    offsets[LLMINT8_WS_OUTLIER_IDX] = L.idx;
    offsets[LLMINT8_WS_ROW_SCALE] = L.row_scale;
    offsets[LLMINT8_WS_CODES] = L.codes;
    return LLMINT8_OK;
}

llmint8_status llmint8_device_status(void* workspace, void* stream) {
    if (!workspace) return LLMINT8_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return LLMINT8_ECUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, workspace, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return LLMINT8_ECUDA;
    if (word != 0 && cudaMemset(workspace, 0, 4) != cudaSuccess) return LLMINT8_ECUDA;
    return static_cast<llmint8_status>(word);
}

size_t llmint8_chain_state_bytes(int M, int N) {
    if (M < 1 || M > kChainMaxM || N < 16 || N > (1 << 30) || (N % 16)) return 0;
    return chain_state_bytes(M, N);
}

llmint8_status llmint8_chain_state_layout(int M, int N, size_t* offsets) {
    if (!offsets || llmint8_chain_state_bytes(M, N) == 0) return LLMINT8_EINVAL;
    offsets[0] = chain_flags_off();
    offsets[1] = chain_parts_off(N);
    offsets[2] = chain_state_bytes(M, N);
    return LLMINT8_OK;
}

// llmint8_matmul_chain and its int32 form (c_out set)
static llmint8_status chain_impl(const void* X, int M, int K, int N, float threshold, const void* state_in,
                          size_t state_in_bytes, const int8_t* Wq, const float* colScaleW, const void* W16, void* Y,
                          float next_threshold, void* state_out, size_t state_out_bytes, int32_t* c_out,
                          void* workspace, size_t workspace_bytes, void* stream) {
    Layout L;
    DeviceInfo* dev = nullptr;
    // with a state in, its flags stand for the threshold (the argument is not used)
    const float t = state_in ? 0.0f : threshold;
    llmint8_status st = check_common(X, M, K, N, t, workspace, workspace_bytes, &L, &dev);
    if (st != LLMINT8_OK) return st;
    if (!Wq || !colScaleW || !Y) return LLMINT8_EINVAL;
    if (state_out && std::isnan(next_threshold)) return LLMINT8_EINVAL;
    if (state_in && state_in == state_out) return LLMINT8_EINVAL;
    const bool use_outliers = !(std::isinf(t) && t > 0);
    if (use_outliers && !W16) return LLMINT8_EINVAL;
    if (!aligned16(Wq) || !aligned16(colScaleW) || !aligned16(Y) || (W16 && !aligned16(W16)) ||
        (state_in && !aligned16(state_in)) || (state_out && !aligned16(state_out)) || (c_out && !aligned16(c_out)))
        return LLMINT8_EALIGN;
    if (!chain_shape_ok(M, K)) return LLMINT8_EUNSUPPORTED;
    // the state buffers must hold the states this call reads and writes
    if (state_in && state_in_bytes < chain_state_bytes(M, K)) return LLMINT8_EINVAL;
    if (state_out && state_out_bytes < chain_state_bytes(M, N)) return LLMINT8_EINVAL;
    if ((st = current_device(&dev)) != LLMINT8_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!state_in && (st = xpass_launch<__half>(X, M, K, threshold, workspace, L, dev, s, W16, N, false)) != LLMINT8_OK)
        return st;
    const WsView w(workspace, L);
    GemvArgs ga;
    ga.codes = reinterpret_cast<const int8_t*>(w.codes);
    ga.Wq = Wq;
    ga.col_scale = colScaleW;
    ga.row_scale = w.row_scale;
    ga.W16 = static_cast<const __half*>(W16);
    ga.hdr = w.hdr;
    ga.outlier_idx = w.idx;
    ga.xo = w.xo;
    ga.xo_pitch = L.kp;
    ga.out = Y;
    ga.M = M;
    ga.K = K;
    ga.N = N;
    ga.use_outliers = use_outliers ? 1 : 0;
    ga.w8 = 0;
    ga.W16c = nullptr;
    ga.row_map = nullptr;
    ga.w16_rows = 0;
    ga.k_per_warp = 0;
    ChainArgs ch;
    ch.X = static_cast<const __half*>(X);
    ch.in = static_cast<const uint8_t*>(state_in);
    ch.out = static_cast<uint8_t*>(state_out);
    ch.next_t = next_threshold;
    ch.err = w.hdr;
    ch.spin_limit = kDefaultSpinLimit;
    ch.c_out = c_out;
    ch.ws_codes = reinterpret_cast<int8_t*>(w.codes);
    ch.ws_row_scale = w.row_scale;
    ch.ws_idx = w.idx;
    ch.ws_count = &w.hdr->outlier_count;
    return chain_launch(ga, ch, dev, s);
}

llmint8_status llmint8_matmul_chain(const void* X, int M, int K, int N, float threshold, const void* state_in,
                                    size_t state_in_bytes, const int8_t* Wq, const float* colScaleW, const void* W16,
                                    void* Y, float next_threshold, void* state_out, size_t state_out_bytes,
                                    void* workspace, size_t workspace_bytes, void* stream) {
    return chain_impl(X, M, K, N, threshold, state_in, state_in_bytes, Wq, colScaleW, W16, Y, next_threshold,
                      state_out, state_out_bytes, nullptr, workspace, workspace_bytes, stream);
}

llmint8_status llmint8_matmul_chain_i32(const void* X, int M, int K, int N, float threshold, const void* state_in,
                                        size_t state_in_bytes, const int8_t* Wq, const float* colScaleW,
                                        const void* W16, void* Y, float next_threshold, void* state_out,
                                        size_t state_out_bytes, int32_t* C, void* workspace, size_t workspace_bytes,
                                        void* stream) {
    if (!C) return LLMINT8_EINVAL;
    return chain_impl(X, M, K, N, threshold, state_in, state_in_bytes, Wq, colScaleW, W16, Y, next_threshold,
                      state_out, state_out_bytes, C, workspace, workspace_bytes, stream);
}

llmint8_status llmint8_selftest_timeout(void* workspace, int spin_limit, void* stream) {
    if (!workspace || spin_limit < 1 || spin_limit > 10000000) return LLMINT8_EINVAL;
    DeviceInfo* dev = nullptr;
    llmint8_status st = current_device(&dev);
    if (st != LLMINT8_OK) return st;
    k_selftest_timeout<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<WsHeader*>(workspace),
                                                                        (uint32_t)spin_limit);
    return launch_status();
}

}  // extern "C"

// ----------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot allocate device memory at the moment they run the matmul:
// callers that must not risk the device-wide synchronization that
// cudaMalloc/cudaFree may cause inside a latency-critical decode loop, hosts
// whose device memory budget is owned by another allocator, and plug-ins that
// are handed device pointers but no allocation rights.  For them the scratch space the
// matmul needs lives in this file-scope array, sized once at load time; every
// GPU that loads the library holds it until the process exits.
// ----------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;  // 8 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
void* g_noalloc_ptr[kMaxDevices];  // device address of g_noalloc_scratch, per device
}  // namespace

extern "C" llmint8_status llmint8_matmul_noalloc(const void* X, int M, int K, int N, float threshold,
                                                 const int8_t* Wq, const float* colScaleW, const void* W16, void* Y, void* stream) {
    if (!sizes_ok(M, K, N)) return LLMINT8_EINVAL;
    if (make_layout(M, K, N).total > kNoAllocScratchBytes) return LLMINT8_EWORKSPACE;
    DeviceInfo* dev = nullptr;
    llmint8_status st = current_device(&dev);
    if (st != LLMINT8_OK) return st;
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return LLMINT8_ECUDA;
    void* scratch = nullptr;
    {
        // one-time set-up per device, with that device current: host code only
        // holds a stand-in for the array, so its device address is looked up
        std::lock_guard<std::mutex> lock(g_mu);
        if (g_noalloc_ptr[d] == nullptr) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return LLMINT8_ECUDA;
            g_noalloc_ptr[d] = p;
        }
        scratch = g_noalloc_ptr[d];
    }
    return llmint8_matmul(X, M, K, N, threshold, Wq, colScaleW, W16, Y, scratch, kNoAllocScratchBytes,
                          stream);
}
