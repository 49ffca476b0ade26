// X pass of the LLM.int8() matmul: outlier-column detection (A1) and per-row
// absmax quantization of the non-outlier columns (A2).
//
//   A1 (paper walkthrough, section 2.3): column j of X is an outlier dimension
//      when some |X[i,j]| exceeds the threshold.
//   A2 (paper walkthrough, sections 2.1 and 2.3; pitfalls guide, section 1):
//      s_x[i] = max over non-outlier j of |X[i,j]|,
//      q = round-half-away(fp32(x * fp32(127 / s_x[i]))), outlier columns -> 0.
//
// The outlier set depends on every row and each row's scale depends on the
// set, so the pass is two kernels: a scan that ORs per-column flags into a bit
// map (atomics only for words that hold an outlier, which is rare), then one
// CTA per row that re-reads its row (from L2 when X fits there) and writes the
// codes: as int8 for the decode GEMV (int8 mma.sync), or as fp16 values (exact
// integers in [-127, 127]) for the tensor-core GEMM (sm_103a has no int8
// tcgen05 kind).
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace llmint8 {

constexpr int kScanThreads = 256;
constexpr int kScanCols = 256;  // columns per CTA: 32 lanes x 8 fp16

// |x| > t for the 8 values (format T) of a 16-byte vector -> 8-bit mask (bit e = element e).
template <typename T>
__device__ __forceinline__ uint32_t outlier_mask8(uint4 v, float t) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t m = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = Fmt<T>::to_float2(w[e]);
        m |= (fabsf(f.x) > t ? 1u : 0u) << (2 * e);
        m |= (fabsf(f.y) > t ? 1u : 0u) << (2 * e + 1);
    }
    return m;
}

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start before its predecessor finishes;
// pdl_wait() blocks until the predecessor has completed and its writes are
// visible (a no-op for a normal launch), pdl_trigger() lets the successor start.
// Every kernel of a call is launched this way, the first one included, so a
// call's kernels (and the weight prefetch of its GEMV) may start while the
// previous call's last kernel drains.  Rule that keeps this safe: before
// pdl_wait() a kernel reads nothing but the weights (constant inputs) and
// writes nothing outside its own shared memory; X and the workspace are
// touched only after it, and through L2 (ld.global.cg), since the
// non-coherent read-only path requires data that no running kernel writes.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// A1.  grid = (ceil(K/256), row groups).  With one row group (gridDim.y == 1)
// every CTA sees all rows of its columns and stores its bitmap words directly;
// with several, the words are OR-ed atomically and the bitmap must be zero on
// entry.  `hdr`, when given, has its error word cleared by CTA 0 (the first
// kernel of a call resets the word).
template <typename T>
__global__ void __launch_bounds__(kScanThreads) k_outlier_scan(const __half* __restrict__ X, int M, int K, float t,
                                                               uint32_t* __restrict__ bitmap, WsHeader* hdr) {
    pdl_trigger();
    if (gridDim.y == 1 && (threadIdx.x & 31) == 0 && blockIdx.x * kScanCols < K) {
        // this CTA's X segments into L2 while the predecessor finishes
        const uint32_t bytes = 2u * (uint32_t)min(kScanCols, K - (int)blockIdx.x * kScanCols);
        for (int r = threadIdx.x >> 5; r < M; r += 8)
            prefetch_l2_bulk(X + (size_t)r * K + (size_t)blockIdx.x * kScanCols, bytes);
    }
    pdl_wait();
    if (hdr != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) hdr->status = 0u;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c0 = blockIdx.x * kScanCols + lane * 8;
    uint32_t m = 0;
    if (c0 < K) {
        const __half* p = X + c0;
        int r = blockIdx.y * 8 + warp;
        const int step = gridDim.y * 8;
        // four independent loads in flight per iteration (a warp walks ~M / (8 gy) rows)
        for (; r + 3 * step < M; r += 4 * step) {
            uint4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) x[u] = ldg_cg_v4(p + (size_t)(r + u * step) * K);
#pragma unroll
            for (int u = 0; u < 4; ++u) m |= outlier_mask8<T>(x[u], t);
        }
        for (; r < M; r += step) m |= outlier_mask8<T>(ldg_cg_v4(p + (size_t)r * K), t);
    }
    // lanes 4w..4w+3 hold the 32 columns of bitmap word w of this strip
    uint32_t word = m << (8 * (lane & 3));
    word |= __shfl_xor_sync(0xffffffffu, word, 1);
    word |= __shfl_xor_sync(0xffffffffu, word, 2);
    __shared__ uint32_t s_words[8][8];
    if ((lane & 3) == 0) s_words[warp][lane >> 2] = word;
    __syncthreads();
    if (threadIdx.x < 8) {
        uint32_t acc = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) acc |= s_words[w][threadIdx.x];
        const int gw = blockIdx.x * (kScanCols / 32) + threadIdx.x;
        if (gw < (K + 31) / 32) {
            if (gridDim.y == 1)
                bitmap[gw] = acc;
            else if (acc != 0u)
                atomicOr(&bitmap[gw], acc);
        }
    }
}

constexpr int kRowThreads = 256;
constexpr int kMaxK = 65536;             // bitmap words held in shared memory: <= 2048
constexpr int kMaxWords = kMaxK / 32;

struct RowQuantArgs {
    const __half* X;
    int M, K;
    const uint32_t* bitmap;   // [ceil(K/32)]
    WsHeader* hdr;            // outlier_count written by block 0
    int32_t* outlier_idx;     // [K], written by block 0
    float* row_scale;         // [M]
    void* codes;              // [M, K]: int8, or fp16 values when codes_fp16
    int codes_fp16;
    __half* xo;               // [M, xo_pitch] gathered outlier columns (nullptr: skip)
    int xo_pitch;             // elements; gathered columns are zero-padded up to a multiple of 64
    int no_outliers;          // threshold +inf: no scan ran, the bit map is not read
    int clear_status;         // no earlier kernel of this call reset the error word
    float t;                  // outlier threshold (cluster_flags)
    // prefill only (k_row_quant_warp): also write the A4 operand of the GEMM,
    // W16oT[n, p] = W16[O[p], n] (zero up to a multiple of 64); skipped if null
    const __half* W16;        // [K, N]
    int N;
    __half* w16o;             // [N, w16o_pitch]
    int w16o_pitch;
    int cluster_flags;        // launched as one cluster of M CTAs: the outlier columns are
                              // found here (no scan kernel, the bit map is not read)
    int rows_per_cta;         // k_row_quant_warp: rows of a CTA (<= 8; its other warps idle)
};

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// Round half away from zero, then clamp to [-127, 127] (clamp after rounding,
// before the integer conversion: LLM quantization in practice, section 3.2).
__device__ __forceinline__ float code_of(float x, float sf) {
    float r = roundf(__fmul_rn(x, sf));
    return fminf(fmaxf(r, -127.0f), 127.0f);
}

// A2.  One CTA per row.  VPT = 16-byte vectors per thread kept in registers
// between the absmax pass and the code pass (the row is re-read when K is
// larger than 256 * 8 * VPT).
//
// Decode with short rows (cluster_flags, VPT 1 or 2): the M CTAs form one thread-block cluster and
// find the outlier columns themselves, without the scan kernel.  Each CTA flags
// the columns of its own row (already in registers), pushes that bit map into
// the shared memory of every CTA of the cluster, and after one cluster barrier
// ORs the M row maps locally (A1: a column is an outlier when any row exceeds t).
template <int VPT, typename T>
__global__ void __launch_bounds__(kRowThreads) k_row_quant(RowQuantArgs a) {
    // bit-map words held in shared memory: the whole row when it sits in registers
    constexpr int kWords = VPT > 0 ? (VPT * 64 > kRowThreads ? VPT * 64 : kRowThreads) : kMaxWords;
    constexpr bool kCluster = VPT == 1 || VPT == 2;     // instantiations that serve cluster_flags
    constexpr int kRowWords = kCluster ? VPT * 64 : 1;  // bit-map words of one row
    __shared__ uint32_t s_bits[kWords];
    __shared__ int32_t s_prefix[kWords];  // outliers in words before w
    __shared__ uint32_t s_rowflags[kCluster ? LLMINT8_DECODE_MAX_M : 1][kRowWords];  // [row][word]
    __shared__ int32_t s_wsum[kRowThreads / 32];
    __shared__ float s_wmax[kRowThreads / 32];
    __shared__ int32_t s_total;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = blockIdx.x;
    const int K = a.K;
    const int nwords = (K + 31) >> 5;
    const bool cflags = kCluster && a.cluster_flags;
    // first half of the barrier that makes sure every CTA of the cluster runs
    // before any writes into its shared memory
    if (cflags) cluster_arrive_relaxed();
    pdl_trigger();
    // this CTA's row of X into L2 while the predecessor finishes (32 KB per request)
    for (int off = tid * 32768; off < 2 * K; off += kRowThreads * 32768)
        prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(a.X + (size_t)row * K) + off, (uint32_t)min(32768, 2 * K - off));
    pdl_wait();

    const __half* xrow = a.X + (size_t)row * K;
    const int nvec = K >> 3;  // K % 16 == 0
    uint4 v[VPT > 0 ? VPT : 1];
    if (VPT > 0) {
#pragma unroll
        for (int i = 0; i < (VPT > 0 ? VPT : 1); ++i) {
            const int vi = tid + i * kRowThreads;
            if (vi < nvec) v[i] = ldg_cg_v4(xrow + (size_t)vi * 8);
        }
    }
    if (a.clear_status && row == 0 && tid == 0) a.hdr->status = 0u;

    if (cflags) {
        namespace cg = cooperative_groups;
        cg::cluster_group cluster = cg::this_cluster();
        const unsigned csize = cluster.num_blocks();  // == M, rank == row
        cluster_wait();
#pragma unroll
        for (int i = 0; i < (VPT > 0 ? VPT : 1); ++i) {
            const int vi = tid + i * kRowThreads;
            // lanes 4k..4k+3 hold the 4 vectors (32 columns) of bit-map word vi / 4
            uint32_t word = (vi < nvec ? outlier_mask8<T>(v[i], a.t) : 0u) << (8 * (lane & 3));
            word |= __shfl_xor_sync(0xffffffffu, word, 1);
            word |= __shfl_xor_sync(0xffffffffu, word, 2);
            if ((lane & 3) == 0 && vi < nvec)
                for (unsigned r = 0; r < csize; ++r) *cluster.map_shared_rank(&s_rowflags[row][vi >> 2], r) = word;
        }
        cluster.sync();  // every row's map has landed everywhere; no remote access follows
    }

    // --- bitmap -> shared memory, exclusive prefix of popcounts (block scan) ---
    constexpr int WPT = kWords / kRowThreads;  // words per thread
    int local[WPT];
    int tsum = 0;
#pragma unroll
    for (int i = 0; i < WPT; ++i) {
        const int w = tid * WPT + i;
        uint32_t b = 0u;
        if (w < nwords && !a.no_outliers) {
            if (cflags) {
                for (int r = 0; r < a.M; ++r) b |= s_rowflags[r][w];
            } else {
                b = __ldcg(a.bitmap + w);
            }
        }
        if (w < nwords) s_bits[w] = b;
        local[i] = __popc(b);
        tsum += local[i];
    }
    int incl = tsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int w = 0; w < kRowThreads / 32; ++w) {
            const int v = s_wsum[w];
            s_wsum[w] = run;
            run += v;
        }
        s_total = run;
    }
    __syncthreads();
    int run = s_wsum[warp] + incl - tsum;
#pragma unroll
    for (int i = 0; i < WPT; ++i) {
        const int w = tid * WPT + i;
        if (w < nwords) s_prefix[w] = run;
        run += local[i];
    }
    __syncthreads();
    const int n_out = s_total;

    // --- masked absmax over the non-outlier columns of this row ---
    float amax = 0.0f;
    auto absmax_vec = [&](uint4 x, int c) {
        const uint32_t om = (s_bits[c >> 5] >> (c & 31)) & 0xFFu;
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = Fmt<T>::to_float2(w[e]);
            if (!((om >> (2 * e)) & 1u)) amax = fmaxf(amax, fabsf(f.x));
            if (!((om >> (2 * e + 1)) & 1u)) amax = fmaxf(amax, fabsf(f.y));
        }
    };
    if (VPT > 0) {
#pragma unroll
        for (int i = 0; i < (VPT > 0 ? VPT : 1); ++i) {
            const int vi = tid + i * kRowThreads;
            if (vi < nvec) absmax_vec(v[i], vi * 8);
        }
    } else {
        for (int vi = tid; vi < nvec; vi += kRowThreads) absmax_vec(ldg_cg_v4(xrow + (size_t)vi * 8), vi * 8);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) s_wmax[warp] = amax;
    __syncthreads();
    amax = s_wmax[0];
#pragma unroll
    for (int w = 1; w < kRowThreads / 32; ++w) amax = fmaxf(amax, s_wmax[w]);

    // scale factor 127 / absmax in fp32, correctly rounded; absmax 0 -> 0
    const float sf = amax > 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;

    // --- codes (outlier columns -> 0) ---
    auto code_vec = [&](uint4 x, int c) {
        const uint32_t om = (s_bits[c >> 5] >> (c & 31)) & 0xFFu;
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        float q[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = Fmt<T>::to_float2(w[e]);
            q[2 * e] = ((om >> (2 * e)) & 1u) ? 0.0f : code_of(f.x, sf);
            q[2 * e + 1] = ((om >> (2 * e + 1)) & 1u) ? 0.0f : code_of(f.y, sf);
        }
        if (a.codes_fp16) {
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                __half2 h = __floats2half2_rn(q[2 * e], q[2 * e + 1]);
                o[e] = *reinterpret_cast<uint32_t*>(&h);
            }
            __half* crow = static_cast<__half*>(a.codes) + (size_t)row * K;
            *reinterpret_cast<uint4*>(crow + c) = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
            uint32_t o[2];
#pragma unroll
            for (int e = 0; e < 2; ++e)
                o[e] = ((uint32_t)(uint8_t)(int8_t)(int)q[4 * e]) | ((uint32_t)(uint8_t)(int8_t)(int)q[4 * e + 1] << 8) |
                       ((uint32_t)(uint8_t)(int8_t)(int)q[4 * e + 2] << 16) |
                       ((uint32_t)(uint8_t)(int8_t)(int)q[4 * e + 3] << 24);
            int8_t* crow = static_cast<int8_t*>(a.codes) + (size_t)row * K;
            *reinterpret_cast<uint2*>(crow + c) = make_uint2(o[0], o[1]);
        }
    };
    if (VPT > 0) {
#pragma unroll
        for (int i = 0; i < (VPT > 0 ? VPT : 1); ++i) {
            const int vi = tid + i * kRowThreads;
            if (vi < nvec) code_vec(v[i], vi * 8);
        }
    } else {
        for (int vi = tid; vi < nvec; vi += kRowThreads) code_vec(ldg_cg_v4(xrow + (size_t)vi * 8), vi * 8);
    }
    if (tid == 0) a.row_scale[row] = amax;

    // --- outlier list (block 0) and gathered outlier columns of this row ---
    if (VPT > 0 && n_out > 0 && (a.xo != nullptr || row == 0)) {
        // from the registers that hold the row: each thread places the outliers
        // of its own vectors
        __half* xo_row = a.xo ? a.xo + (size_t)row * a.xo_pitch : nullptr;
#pragma unroll
        for (int i = 0; i < (VPT > 0 ? VPT : 1); ++i) {
            const int vi = tid + i * kRowThreads;
            if (vi < nvec) {
                const int w = vi >> 2, sh = (vi & 3) * 8;
                const uint32_t word = s_bits[w];
                uint32_t b = (word >> sh) & 0xFFu;
                while (b) {
                    const int e = __ffs(b) - 1;
                    b &= b - 1;
                    const int pos = s_prefix[w] + __popc(word & ((1u << (sh + e)) - 1u));
                    if (xo_row) {
                        const uint4 x = v[i];
                        const uint32_t w32 = (e & 4) ? ((e & 2) ? x.w : x.z) : ((e & 2) ? x.y : x.x);
                        xo_row[pos] = __ushort_as_half((unsigned short)(w32 >> (16 * (e & 1))));
                    }
                    if (row == 0) a.outlier_idx[pos] = 8 * vi + e;
                }
            }
        }
    } else if (n_out > 0 && (a.xo != nullptr || row == 0)) {
        __half* xo_row = a.xo ? a.xo + (size_t)row * a.xo_pitch : nullptr;
        for (int w = tid; w < nwords; w += kRowThreads) {
            uint32_t b = s_bits[w];
            int pos = s_prefix[w];
            while (b) {
                const int bit = __ffs(b) - 1;
                b &= b - 1;
                const int col = w * 32 + bit;
                if (xo_row) xo_row[pos] = __ldcg(xrow + col);
                if (row == 0) a.outlier_idx[pos] = col;
                ++pos;
            }
        }
    }
    if (a.xo != nullptr) {
        // zero padding up to the next multiple of 64 gathered columns
        __half* xo_row = a.xo + (size_t)row * a.xo_pitch;
        const int padded = (n_out + 63) & ~63;
        for (int c = n_out + tid; c < padded; c += kRowThreads) xo_row[c] = __ushort_as_half(0);
    }
    if (row == 0 && tid == 0) a.hdr->outlier_count = n_out;
}

// A2 for many rows of at most 256 * VPL columns (prefill): one warp per row,
// up to 8 rows per CTA (fewer when that spreads the rows evenly: two CTAs fit
// on an SM, and 256 CTAs of 8 rows on 148 SMs would give 108 SMs twice the rows
// of the other 40).  The CTA reads the outlier bit map and forms its prefix once
// for its 8 rows; each warp holds its row in registers (VPL 16-byte vectors
// per lane), reduces the masked absmax with shuffles, writes the codes and
// places its outlier values from the same registers.  No barrier sits between
// the loads of a row and its codes, where the one-CTA-per-row kernel had four.
//
// With w16o set, the CTAs also write the A4 operand of the tensor-core GEMM,
// W16oT[n, p] = W16[O[p], n] (zero for count <= p < a multiple of 64), each CTA
// a share of the 16-column groups of N, through a shared-memory transpose: the
// outlier list is already here, so no separate gather launch is needed.
constexpr int kRowsPerCta = 8;
constexpr int kGatherCols = 16;

template <int VPL, typename T>
__global__ void __launch_bounds__(kRowsPerCta * 32) k_row_quant_warp(RowQuantArgs a) {
    constexpr int kWords = 8 * VPL;  // bit-map words of a row (<= the CTA's 256 threads)
    static_assert(kWords <= kRowsPerCta * 32, "one bit-map word per thread");
    __shared__ uint32_t s_bits[kWords];
    __shared__ int32_t s_prefix[kWords];
    __shared__ int32_t s_wsum[kRowsPerCta];
    __shared__ int32_t s_total;
    __shared__ int32_t s_idx[32 * kWords];                    // the outlier list, for the gather
    __shared__ __align__(16) __half s_tile[64][kGatherCols];  // 64 outliers x 16 columns

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = blockIdx.x * a.rows_per_cta + warp;
    const bool live = warp < a.rows_per_cta && row < a.M;
    const int K = a.K;
    const int nwords = (K + 31) >> 5;
    const int nvec = K >> 3;  // K % 16 == 0
    pdl_trigger();
    pdl_wait();

    const __half* xrow = a.X + (size_t)(live ? row : 0) * K;
    uint4 v[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int vi = lane + 32 * i;
        v[i] = (live && vi < nvec) ? ldg_cg_v4(xrow + (size_t)vi * 8) : make_uint4(0, 0, 0, 0);
    }
    if (a.clear_status && blockIdx.x == 0 && tid == 0) a.hdr->status = 0u;

    // --- bit map -> shared memory, exclusive prefix of popcounts (one word per thread) ---
    const uint32_t b = (tid < nwords && !a.no_outliers) ? __ldcg(a.bitmap + tid) : 0u;
    if (tid < kWords) s_bits[tid] = b;
    const int cnt = __popc(b);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int w = 0; w < kRowsPerCta; ++w) {
            const int y = s_wsum[w];
            s_wsum[w] = run;
            run += y;
        }
        s_total = run;
    }
    __syncthreads();
    const bool gather = a.w16o != nullptr;
    if (tid < kWords) {
        const int pre = s_wsum[warp] + incl - cnt;
        s_prefix[tid] = pre;
        if (gather) {  // positions of this word's outliers in the list
            uint32_t bb = b;
            for (int k = pre; bb; ++k) {
                s_idx[k] = 32 * tid + __ffs(bb) - 1;
                bb &= bb - 1;
            }
        }
    }
    __syncthreads();
    const int n_out = s_total;

    // --- this warp's row ---
    if (live) {
        // masked absmax over the non-outlier columns
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int c = 8 * (lane + 32 * i);
            if (c < K) {
                const uint32_t om = (s_bits[c >> 5] >> (c & 31)) & 0xFFu;
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = Fmt<T>::to_float2(w[e]);
                    if (!((om >> (2 * e)) & 1u)) amax = fmaxf(amax, fabsf(f.x));
                    if (!((om >> (2 * e + 1)) & 1u)) amax = fmaxf(amax, fabsf(f.y));
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        // scale factor 127 / absmax in fp32, correctly rounded; absmax 0 -> 0
        const float sf = amax > 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
        if (lane == 0) a.row_scale[row] = amax;

        // codes (outlier columns -> 0), outlier values and list from the registers
        __half* xo_row = (a.xo != nullptr && n_out > 0) ? a.xo + (size_t)row * a.xo_pitch : nullptr;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int vi = lane + 32 * i, c = 8 * vi;
            if (c >= K) continue;
            const int wd = c >> 5, sh = c & 31;
            const uint32_t word = s_bits[wd];
            const uint32_t om = (word >> sh) & 0xFFu;
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            float q[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = Fmt<T>::to_float2(w[e]);
                q[2 * e] = ((om >> (2 * e)) & 1u) ? 0.0f : code_of(f.x, sf);
                q[2 * e + 1] = ((om >> (2 * e + 1)) & 1u) ? 0.0f : code_of(f.y, sf);
            }
            if (a.codes_fp16) {
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    __half2 h = __floats2half2_rn(q[2 * e], q[2 * e + 1]);
                    o[e] = *reinterpret_cast<uint32_t*>(&h);
                }
                *reinterpret_cast<uint4*>(static_cast<__half*>(a.codes) + (size_t)row * K + c) =
                    make_uint4(o[0], o[1], o[2], o[3]);
            } else {
                uint32_t o[2];
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    o[e] = ((uint32_t)(uint8_t)(int8_t)(int)q[4 * e]) |
                           ((uint32_t)(uint8_t)(int8_t)(int)q[4 * e + 1] << 8) |
                           ((uint32_t)(uint8_t)(int8_t)(int)q[4 * e + 2] << 16) |
                           ((uint32_t)(uint8_t)(int8_t)(int)q[4 * e + 3] << 24);
                *reinterpret_cast<uint2*>(static_cast<int8_t*>(a.codes) + (size_t)row * K + c) =
                    make_uint2(o[0], o[1]);
            }
            uint32_t bits = om;
            while (bits) {
                const int e = __ffs(bits) - 1;
                bits &= bits - 1;
                const int pos = s_prefix[wd] + __popc(word & ((1u << (sh + e)) - 1u));
                if (xo_row) {
                    const uint32_t w32 = (e & 4) ? ((e & 2) ? w[3] : w[2]) : ((e & 2) ? w[1] : w[0]);
                    xo_row[pos] = __ushort_as_half((unsigned short)(w32 >> (16 * (e & 1))));
                }
                if (row == 0) a.outlier_idx[pos] = c + e;
            }
        }
        if (a.xo != nullptr) {
            // zero padding up to the next multiple of 64 gathered columns
            __half* xr = a.xo + (size_t)row * a.xo_pitch;
            const int padded = (n_out + 63) & ~63;
            for (int c = n_out + lane; c < padded; c += 32) xr[c] = __ushort_as_half(0);
        }
        if (row == 0 && lane == 0) a.hdr->outlier_count = n_out;
    }

    // --- A4 operand of the GEMM: W16oT for this CTA's 16-column groups ---
    if (gather && n_out > 0) {
        const int padded = (n_out + 63) & ~63;
        const int groups = a.N / kGatherCols;
        for (int gp = blockIdx.x; gp < groups; gp += gridDim.x) {
            const int n0 = gp * kGatherCols;
            for (int p0 = 0; p0 < padded; p0 += 64) {
                {   // read: outlier p0 + p, columns n0 + 4j .. +3 (8 bytes of one W16 row)
                    const int p = tid >> 2, j = (tid & 3) * 4;
                    uint2 val = make_uint2(0u, 0u);
                    if (p0 + p < n_out)
                        val = *reinterpret_cast<const uint2*>(a.W16 + (size_t)s_idx[p0 + p] * a.N + n0 + j);
                    *reinterpret_cast<uint2*>(&s_tile[p][j]) = val;
                }
                __syncthreads();
                {   // write: row n0 + jn of W16oT, outliers p0 + 4q .. +3
                    const int jn = tid >> 4, q4 = (tid & 15) * 4;
                    const uint32_t lo = (uint32_t)__half_as_ushort(s_tile[q4][jn]) |
                                        ((uint32_t)__half_as_ushort(s_tile[q4 + 1][jn]) << 16);
                    const uint32_t hi = (uint32_t)__half_as_ushort(s_tile[q4 + 2][jn]) |
                                        ((uint32_t)__half_as_ushort(s_tile[q4 + 3][jn]) << 16);
                    *reinterpret_cast<uint2*>(a.w16o + (size_t)(n0 + jn) * a.w16o_pitch + p0 + q4) =
                        make_uint2(lo, hi);
                }
                __syncthreads();
            }
        }
    }
}

// A4 operand preparation for the tensor-core GEMM: W16oT[n, p] = W16[O[p], n]
// for p < count, zero for count <= p < roundup(count, 64).  W16 is [K, N]
// row-major; the result is [N, pitch] with the gathered K contiguous, the
// K-major layout the MMA reads.  grid.x = ceil(N / 64); 256 threads.
// W8Rows: the A4 operand when no full fp16 copy of W is kept (W16 is then
// nullptr): row k is W16c[row_map[k]] if 0 <= row_map[k] < rows, else the
// dequantized codes Wq[n, k] with colScaleW[n].
struct W8Rows {
    const __half* W16c;
    const int32_t* row_map;
    int rows;
    const int8_t* Wq;  // [N, K]
    int K;
    const float* col_scale;
};

template <typename T>
__global__ void __launch_bounds__(256) k_gather_w16_outlier_rows(const __half* __restrict__ W16, int N,
                                                                 const WsHeader* __restrict__ hdr,
                                                                 const int32_t* __restrict__ outlier_idx,
                                                                 __half* __restrict__ w16oT, int pitch, W8Rows w8) {
    __shared__ __half tile[64][64 + 8];
    pdl_trigger();
    pdl_wait();
    const int count = __ldcg(&hdr->outlier_count);
    const int padded = (count + 63) & ~63;
    const int n0 = blockIdx.x * 64;
    const int tid = threadIdx.x;
    for (int p0 = 0; p0 < padded; p0 += 64) {
        // load 64 gathered rows x 64 columns (coalesced along n)
        for (int e = tid; e < 64 * 64; e += 256) {
            const int pr = e >> 6, nc = e & 63;
            const int p = p0 + pr, n = n0 + nc;
            __half v = __ushort_as_half(0);
            if (p < count && n < N) {
                const int k = __ldcg(outlier_idx + p);
                if (W16 != nullptr) {
                    v = W16[(size_t)k * N + n];
                } else {
                    const int rm = w8.row_map != nullptr ? __ldg(w8.row_map + k) : -1;
                    v = (rm >= 0 && rm < w8.rows) ? w8.W16c[(size_t)rm * N + n]
                                                  : dequant_weight<T>(w8.Wq[(size_t)n * w8.K + k], w8.col_scale[n]);
                }
            }
            tile[pr][nc] = v;
        }
        __syncthreads();
        // write transposed: row n, columns p0..p0+63 (coalesced along p)
        for (int e = tid; e < 64 * 64; e += 256) {
            const int nr = e >> 6, pc = e & 63;
            const int n = n0 + nr;
            if (n < N) w16oT[(size_t)n * pitch + p0 + pc] = tile[pc][nr];
        }
        __syncthreads();
    }
}

}  // namespace llmint8
