// Decode chain: a layer's GEMV also prepares the next layer's X pass.
//
// In a decode step every matmul starts with the X pass of its input (A1, A2),
// short kernels whose latency sits between the previous layer's GEMV and this
// one; per-forward conversion of the activations is the cost the LLM.int8()
// paper walkthrough (section 5.4, small-batch performance) holds responsible
// for the method's slowdown at small batch.  When the output Y of a GEMV is the next
// layer's X, the GEMV's epilogue here computes what the next X pass would have
// found from Y:
//   * the outlier flags of Y's columns (A1: some row has |Y[i, j]| > t'), and
//   * per row of Y, the absmax over the columns that are not outliers (the row
//     scale of A2), as one partial maximum per 16-column strip.
// The GEMV holds all M rows of its 16 columns, so both are exact per strip.  The
// next layer's GEMV then runs no X pass: each CTA takes the flags and partial
// maxima (the "chain state"), forms the row scales, and converts its own copy
// of X into codes in shared memory while its first weight tiles arrive.
//
// The kernel is a streaming GEMV for up to 4 rows of X:
//  * one producer thread moves 16 x 512-byte tiles of Wq (16 output columns,
//    512 K; two 2D TMA boxes of 256 K) into an 8-stage mbarrier ring.  The
//    first ring round is requested before griddepcontrol.wait (weights do not
//    depend on the previous kernel).  Without a chain state in, the producer
//    then copies the X codes of the X pass (M x K bytes) into shared memory.
//  * 8 consumer warps: warp w owns columns n0 + 2w and n0 + 2w + 1 of each
//    16-column strip over all of K.  Lane l takes the 16 bytes at offset 16 l
//    of the stage (lanes 0-15 the first box, 16-31 the second) for both columns
//    and the matching 16 bytes of each row of codes, with dp4a (four int8
//    products summed into an exact int32 per instruction).
//  * each strip ends in a warp-local epilogue: the int32 lane partials are
//    summed with redux.sync (exact), the fp16 outlier slice (A4) is spread over
//    the lanes (32 / M lanes per row of X, fp32 products) and summed with
//    shuffles, one lane per row applies the scales (A5) and writes Y, and the
//    chain state of Y is written (flags by each warp; the 8 warps' row maxima
//    are combined by warp 0 through two mbarriers).
// The grid is persistent (CTA b takes strips b, b + G, ...).  Every wait is
// bounded: on a timeout the error word is set, the other roles leave through
// the abort flag, and the producer waits for its copies in flight before the
// CTA ends.
#pragma once

#include "common.cuh"
#include "gemv.cuh"
#include "xpass.cuh"

namespace llmint8 {

constexpr int kChainMaxM = 4;
constexpr int kChainWarps = 8;                           // consumer warps
constexpr int kChainThreads = (kChainWarps + 1) * 32;    // + one producer warp
constexpr int kChainCols = 2 * kChainWarps;              // columns of a strip
constexpr int kChainBoxK = 256;                          // K bytes of one TMA box
constexpr int kChainStageK = 2 * kChainBoxK;             // K of one ring stage
constexpr int kChainBox = kChainCols * kChainBoxK;       // 4 KB
constexpr int kChainStage = 2 * kChainBox;               // 8 KB
constexpr int kChainStages = 8;
constexpr int kChainPre = 2;             // outlier positions per lane held in registers
constexpr int kChainBatch = 4;           // outlier positions per lane loaded together past those
constexpr uint32_t kChainBulk = 32768;   // bytes per bulk copy of the X codes

// Chain state of an activation [M, N] (device memory):
//   header (256 B) | flags: uint8 [N], 1 = outlier column (padded to 256 B) |
//   partial row maxima: float [nparts][M] (absmax of each row over the
//   non-outlier columns of one part of the columns; the row scale is their max).
struct ChainHeader {
    int32_t M, N, nparts;
    float threshold;
    int32_t pad[60];
};
static_assert(sizeof(ChainHeader) == 256, "chain header is 256 bytes");
__host__ __device__ constexpr size_t chain_flags_off() { return sizeof(ChainHeader); }
__host__ __device__ constexpr size_t chain_parts_off(int N) {
    return sizeof(ChainHeader) + ((size_t)N + 255) / 256 * 256;
}
__host__ __device__ constexpr size_t chain_state_bytes(int M, int N) {
    return chain_parts_off(N) + (size_t)(N / kChainCols) * M * 4;
}

struct ChainArgs {
    const __half* X;       // [M, K] X itself (read with a chain state in)
    const uint8_t* in;     // chain state of X, or nullptr (codes from the X pass)
    uint8_t* out;          // chain state of Y to write, or nullptr
    float next_t;          // threshold the flags of Y are taken for
    WsHeader* err;         // error word
    uint32_t spin_limit;   // poll budget of the bounded waits
    int32_t* c_out;        // [M, N] exact int32 accumulator of A3, or nullptr
    // workspace fields of the X pass: with a chain state in, CTA 0 leaves there
    // what it derived (the same fields an X pass fills)
    int8_t* ws_codes;      // [M, K]
    float* ws_row_scale;   // [M]
    int32_t* ws_idx;       // [K] outlier columns, ascending
    int32_t* ws_count;     // outlier count
};

constexpr uint32_t kStatusInvalid = 1;  // == LLMINT8_EINVAL: a chain state that does not fit the call

struct ChainBars {
    uint64_t full[kChainStages];
    uint64_t empty[kChainStages];
    uint64_t xbar;
    uint64_t strip_done[2];  // the 8 warps' row maxima of a strip are in shared memory
    uint64_t strip_free[2];  // warp 0 has combined them
    uint32_t abort_flag;
};

__host__ __device__ constexpr size_t chain_xbytes(int M, int K) { return ((size_t)M * K + 15) / 16 * 16; }
__host__ __device__ constexpr size_t chain_words(int K) { return ((size_t)K + 31) / 32; }
// dynamic shared memory: 1 KB alignment slack, the ring, the codes, the bit map
// and its prefix counts, the barriers
__host__ __device__ constexpr size_t chain_smem(int M, int K) {
    return 1024 + (size_t)kChainStages * kChainStage + chain_xbytes(M, K) + 8 * chain_words(K) + sizeof(ChainBars);
}

__device__ __forceinline__ void chain_bulk_load(void* smem_dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(smem_dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ uint32_t chain_ldg_nc_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
// barrier of the 8 consumer warps only (the producer warp does not take part)
__device__ __forceinline__ void chain_consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// four 0/1 flag bytes -> four bits
__device__ __forceinline__ uint32_t flag_bits4(uint32_t x) {
    return (x & 1u) | ((x >> 7) & 2u) | ((x >> 14) & 4u) | ((x >> 21) & 8u);
}

template <int MR, bool IN_RAW, bool EMIT>
__global__ void __launch_bounds__(kChainThreads, 2)
    k_gemv_chain(const __grid_constant__ CUtensorMap tw, GemvArgs a, ChainArgs ch) {
    constexpr int S = kChainStages;
    constexpr int MP = MR == 1 ? 1 : (MR == 2 ? 2 : 4);  // rows of X rounded up to a power of two
    constexpr int LPR = 32 / MP;                           // lanes per row of X in the outlier slice
    __shared__ float s_part[2][kChainWarps][MR];           // row maxima of Y per warp (EMIT)
    __shared__ float s_wmax[kChainWarps][MR];
    __shared__ float s_sx[MR];
    __shared__ int32_t s_wsum[kChainWarps];
    __shared__ int32_t s_total;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int K = a.K, N = a.N;
    const int nwords = (int)chain_words(K);
    uint8_t* ring = smem;
    int8_t* xs = reinterpret_cast<int8_t*>(smem + S * kChainStage);
    uint32_t* s_bits = reinterpret_cast<uint32_t*>(smem + S * kChainStage + chain_xbytes(MR, K));
    int32_t* s_prefix = reinterpret_cast<int32_t*>(s_bits + nwords);
    ChainBars* sb = reinterpret_cast<ChainBars*>(s_prefix + nwords);
    volatile uint32_t* abort_flag = &sb->abort_flag;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int strips = N / kChainCols, G = gridDim.x;
    const int my_strips = (int)blockIdx.x < strips ? (strips - (int)blockIdx.x + G - 1) / G : 0;
    const int sps = (K + kChainStageK - 1) / kChainStageK;  // ring stages per strip
    const int total = my_strips * sps;

    pdl_trigger();
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&sb->full[s], 1);
            mbar_init(&sb->empty[s], kChainWarps);
        }
        mbar_init(&sb->xbar, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sb->strip_done[b], kChainWarps);
            mbar_init(&sb->strip_free[b], 1);
        }
        sb->abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tw);
    }
    __syncthreads();
    auto fail = [&](uint32_t where) {
        *abort_flag = 1u;
        record_error(ch.err, kStatusTimeout, where);
    };

    if (warp == kChainWarps) {
        // ---------------------------------------------------------------- producer
        if (lane != 0) return;
        const uint32_t xbytes = (uint32_t)(MR * K);
        bool x_issued = false;
        auto issue_x = [&]() {
            pdl_wait();  // the codes are written by the X pass
            if (!IN_RAW) {
                mbar_arrive_expect_tx(&sb->xbar, xbytes);
                for (uint32_t off = 0; off < xbytes; off += kChainBulk)
                    chain_bulk_load(xs + off, a.codes + off, min(kChainBulk, xbytes - off), &sb->xbar);
            }
            x_issued = true;
        };
        uint32_t issued = 0, issued_par = 0;  // per stage: filled at least once, parity of its last fill
        int q = 0, j = 0, st = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int t = 0; t < total; ++t) {
            if (t == S) issue_x();
            // stages of the first round are free; later ones wait for the 8 consumer warps
            if (t >= S && !mbar_wait_bounded(&sb->empty[q], ph ^ 1u, ch.spin_limit, abort_flag)) {
                if (!*abort_flag) fail(21);  // a wait that ran out, not consumers that left
                ok = false;
                break;
            }
            const int n0 = ((int)blockIdx.x + j * G) * kChainCols;
            const int k0 = st * kChainStageK;
            const bool two = k0 + kChainBoxK < K;  // the second box holds columns inside K
            mbar_arrive_expect_tx(&sb->full[q], two ? 2u * kChainBox : (uint32_t)kChainBox);
            tma_load_2d(ring + q * kChainStage, &tw, &sb->full[q], k0, n0);
            if (two) tma_load_2d(ring + q * kChainStage + kChainBox, &tw, &sb->full[q], k0 + kChainBoxK, n0);
            issued |= 1u << q;
            issued_par = (issued_par & ~(1u << q)) | (ph << q);
            if (++q == S) q = 0, ph ^= 1u;
            if (++st == sps) st = 0, ++j;
        }
        if (!x_issued) issue_x();
        // no copy may still target shared memory when the CTA ends, whether the
        // consumers finished or left early: wait for the last fill of every stage
        // (already complete on the normal path) and for the codes
        for (int s = 0; s < S; ++s)
            if ((issued >> s) & 1u) mbar_wait_bounded(&sb->full[s], (issued_par >> s) & 1u, 1u << 20, nullptr);
        if (!IN_RAW) mbar_wait_bounded(&sb->xbar, 0, 1u << 20, nullptr);
        (void)ok;
        return;
    }

    // -------------------------------------------------------------------- consumers
    const int kl = 16 * (lane & 15), bx = lane >> 4;
    const int woff = bx * kChainBox + 2 * warp * kChainBoxK + kl;  // column n0 + 2w, this lane's 16 bytes
    const int oi = lane / LPR, oj = lane % LPR;                    // outlier slice: row of X, first position
    const bool orow = oi < MR;
    auto wait_warp = [&](uint64_t* bar, uint32_t par, uint32_t where) -> bool {
        const bool got = mbar_wait_bounded(bar, par, ch.spin_limit, abort_flag);
        if (__all_sync(0xffffffffu, got)) return true;
        if (lane == 0) fail(where);
        return false;
    };

    pdl_wait();  // everything below may read the previous kernel's results
    const bool outl = a.use_outliers != 0;
    int cnt = 0;
    if (IN_RAW) {
        // ---- the X pass from the chain state: bit map, its prefix counts, row
        // scales, and the codes of X into shared memory ----
        const uint8_t* flags = ch.in + chain_flags_off();
        const float* parts = reinterpret_cast<const float*>(ch.in + chain_parts_off(K));
        // the header must describe an activation of this call's shape: M rows,
        // K columns, and at most one partial maximum per 16-column strip (the
        // host checked that the buffer holds that many); nothing else of the
        // state is read otherwise
        if (blockIdx.x == 0 && tid == 0) ch.err->status = 0u;  // no X pass ran to clear the error word
        const ChainHeader* hin = reinterpret_cast<const ChainHeader*>(ch.in);
        const int hM = ldg_cg_s32(&hin->M), hN = ldg_cg_s32(&hin->N);
        const int nparts = ldg_cg_s32(&hin->nparts);
        if (hM != MR || hN != K || nparts < 1 || nparts > K / kChainCols) {
            // every CTA leaves; CTA 0 alone records it, after clearing the word
            // above, so no earlier write can hide it (the producers, stopped by
            // the flag, record nothing)
            if (tid == 0) {
                if (blockIdx.x == 0) record_error(ch.err, kStatusInvalid, 26);
                *abort_flag = 1u;
            }
            return;
        }
        // bit-map words: each thread takes a contiguous run of words
        const int wpt = (nwords + kChainWarps * 32 - 1) / (kChainWarps * 32);
        const int w0 = min(nwords, tid * wpt), w1 = min(nwords, w0 + wpt);
        int tsum = 0;
        for (int w = w0; w < w1; ++w) {
            uint32_t b = 0u;
            if (outl) {
                const uint4 f0 = ldg_cg_v4(flags + 32 * w);
                const uint4 f1 = 32 * w + 16 < K ? ldg_cg_v4(flags + 32 * w + 16) : make_uint4(0, 0, 0, 0);
                b = flag_bits4(f0.x) | (flag_bits4(f0.y) << 4) | (flag_bits4(f0.z) << 8) | (flag_bits4(f0.w) << 12) |
                    (flag_bits4(f1.x) << 16) | (flag_bits4(f1.y) << 20) | (flag_bits4(f1.z) << 24) |
                    (flag_bits4(f1.w) << 28);
            }
            s_bits[w] = b;
            tsum += __popc(b);
        }
        // row scales: the maxima of the partial maxima
        float pm[MR];
#pragma unroll
        for (int i = 0; i < MR; ++i) pm[i] = 0.0f;
        for (int p = tid; p < nparts; p += kChainWarps * 32)
#pragma unroll
            for (int i = 0; i < MR; ++i) pm[i] = fmaxf(pm[i], __ldcg(parts + (size_t)p * MR + i));
#pragma unroll
        for (int i = 0; i < MR; ++i) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) pm[i] = fmaxf(pm[i], __shfl_xor_sync(0xffffffffu, pm[i], o));
            if (lane == 0) s_wmax[warp][i] = pm[i];
        }
        int incl = tsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) s_wsum[warp] = incl;
        chain_consumer_sync();
        if (tid == 0) {
            int run = 0;
            for (int w = 0; w < kChainWarps; ++w) {
                const int v = s_wsum[w];
                s_wsum[w] = run;
                run += v;
            }
            s_total = run;
        }
        if (tid < MR) {
            float m = s_wmax[0][tid];
            for (int w = 1; w < kChainWarps; ++w) m = fmaxf(m, s_wmax[w][tid]);
            s_sx[tid] = m;
        }
        chain_consumer_sync();
        int run = s_wsum[warp] + incl - tsum;
        for (int w = w0; w < w1; ++w) {
            s_prefix[w] = run;
            run += __popc(s_bits[w]);
        }
        cnt = s_total;
        // codes (outlier columns -> 0), scale factor 127 / absmax as in the X pass
        const int vpr = K >> 3;  // 8-element vectors per row
#pragma unroll
        for (int i = 0; i < MR; ++i) {
            const float amax = s_sx[i];
            const float sf = amax > 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
            for (int c = 8 * tid; c < 8 * vpr; c += 8 * kChainWarps * 32) {
                const uint4 x = ldg_cg_v4(ch.X + (size_t)i * K + c);
                const uint32_t om = (s_bits[c >> 5] >> (c & 31)) & 0xFFu;
                const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
                uint32_t o[2] = {0u, 0u};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wv[e]));
                    const int q0 = ((om >> (2 * e)) & 1u) ? 0 : (int)code_of(f.x, sf);
                    const int q1 = ((om >> (2 * e + 1)) & 1u) ? 0 : (int)code_of(f.y, sf);
                    o[e >> 1] |= (((uint32_t)(uint8_t)(int8_t)q0) | ((uint32_t)(uint8_t)(int8_t)q1 << 8)) << (16 * (e & 1));
                }
                *reinterpret_cast<uint2*>(xs + (size_t)i * K + c) = make_uint2(o[0], o[1]);
            }
        }
        chain_consumer_sync();  // codes, bit map and prefix counts visible to all consumer warps
        if (blockIdx.x == 0) {
            // what this call derived, into the workspace fields an X pass fills
            for (int c = 16 * tid; c < MR * K; c += 16 * kChainWarps * 32)
                *reinterpret_cast<uint4*>(ch.ws_codes + c) = *reinterpret_cast<const uint4*>(xs + c);
            if (tid < MR) ch.ws_row_scale[tid] = s_sx[tid];
            for (int w = w0; w < w1; ++w) {
                uint32_t b = s_bits[w];
                int pos = s_prefix[w];
                while (b) {
                    ch.ws_idx[pos++] = 32 * w + __ffs(b) - 1;
                    b &= b - 1;
                }
            }
            if (tid == 0) *ch.ws_count = s_total;
        }
    } else {
        cnt = outl ? ldg_cg_s32(&a.hdr->outlier_count) : 0;
    }
    // the j-th outlier column: from the list of the X pass, or found in the bit
    // map (last word whose prefix count is <= j, then the matching set bit)
    auto outlier_col = [&](int jo) -> int {
        if (!IN_RAW) return ldg_cg_s32(a.outlier_idx + jo);
        int lo = 0, hi = nwords - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_prefix[mid] <= jo)
                lo = mid;
            else
                hi = mid - 1;
        }
        uint32_t b = s_bits[lo];
        for (int r = jo - s_prefix[lo]; r > 0; --r) b &= b - 1;
        return 32 * lo + __ffs(b) - 1;
    };
    auto outlier_x = [&](int i, int jo, int k) -> uint32_t {
        if (!IN_RAW)
            return (uint32_t)__ldcg(reinterpret_cast<const unsigned short*>(a.xo) + (size_t)i * a.xo_pitch + jo);
        return (uint32_t)__ldcg(reinterpret_cast<const unsigned short*>(ch.X) + (size_t)i * K + k);
    };
    // outlier positions oj + LPR m (m < kChainPre) of this lane: columns and X values
    int kidx[kChainPre];
    uint32_t xraw[kChainPre];
#pragma unroll
    for (int m = 0; m < kChainPre; ++m) {
        const int jo = oj + LPR * m;
        kidx[m] = (outl && jo < cnt) ? outlier_col(jo) : 0;
        xraw[m] = (outl && orow && jo < cnt) ? outlier_x(oi, jo, kidx[m]) : 0u;
    }
    const float rs = orow ? (IN_RAW ? s_sx[oi] : __ldcg(a.row_scale + oi)) : 0.0f;
    if (!IN_RAW && !wait_warp(&sb->xbar, 0, 22)) return;

    float* parts_out = EMIT ? reinterpret_cast<float*>(ch.out + chain_parts_off(N)) : nullptr;
    if (EMIT && blockIdx.x == 0 && tid == 0) {
        ChainHeader* h = reinterpret_cast<ChainHeader*>(ch.out);
        h->M = MR;
        h->N = N;
        h->nparts = strips;
        h->threshold = ch.next_t;
    }

    int q = 0;
    uint32_t ph = 0;
    for (int j = 0; j < my_strips; ++j) {
        const int strip = (int)blockIdx.x + j * G;
        const int nA = strip * kChainCols + 2 * warp;
        // epilogue operands of this strip (constant inputs), in flight during the strip
        const float cs0 = __ldg(a.col_scale + nA), cs1 = __ldg(a.col_scale + nA + 1);
        uint32_t wraw[kChainPre];
#pragma unroll
        for (int m = 0; m < kChainPre; ++m) {
            const int jo = oj + LPR * m;
            wraw[m] = (outl && !a.w8 && orow && jo < cnt) ? chain_ldg_nc_u32(a.W16 + (size_t)kidx[m] * N + nA) : 0u;
        }

        int acc0[MR], acc1[MR];
#pragma unroll
        for (int i = 0; i < MR; ++i) acc0[i] = acc1[i] = 0;
        for (int st = 0; st < sps; ++st) {
            if (!wait_warp(&sb->full[q], ph, 23)) return;
            const int kofs = st * kChainStageK + bx * kChainBoxK + kl;  // K of this lane's 16 bytes
            if (kofs < K) {
                const uint8_t* w = ring + q * kChainStage + woff;
                const uint4 wa = *reinterpret_cast<const uint4*>(w);
                const uint4 wb = *reinterpret_cast<const uint4*>(w + kChainBoxK);
#pragma unroll
                for (int i = 0; i < MR; ++i) {
                    const uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)i * K + kofs);
                    acc0[i] = __dp4a((int)wa.x, (int)xv.x, acc0[i]);
                    acc0[i] = __dp4a((int)wa.y, (int)xv.y, acc0[i]);
                    acc0[i] = __dp4a((int)wa.z, (int)xv.z, acc0[i]);
                    acc0[i] = __dp4a((int)wa.w, (int)xv.w, acc0[i]);
                    acc1[i] = __dp4a((int)wb.x, (int)xv.x, acc1[i]);
                    acc1[i] = __dp4a((int)wb.y, (int)xv.y, acc1[i]);
                    acc1[i] = __dp4a((int)wb.z, (int)xv.z, acc1[i]);
                    acc1[i] = __dp4a((int)wb.w, (int)xv.w, acc1[i]);
                }
            }
            __syncwarp();  // every lane has read the stage
            if (lane == 0) mbar_arrive(&sb->empty[q]);
            if (++q == S) q = 0, ph ^= 1u;
        }

        // A3 sums over the 32 lanes (exact), then this lane's row of X
        int c0 = 0, c1 = 0;
#pragma unroll
        for (int i = 0; i < MR; ++i) {
            const int s0 = __reduce_add_sync(0xffffffffu, acc0[i]);
            const int s1 = __reduce_add_sync(0xffffffffu, acc1[i]);
            if (oi == i) c0 = s0, c1 = s1;
        }
        // A4: positions oj, oj + LPR, ... of the outlier list, summed over the row's lanes
        float f0 = 0.0f, f1 = 0.0f;
        if (cnt > 0) {
#pragma unroll
            for (int m = 0; m < kChainPre; ++m) {
                const int jo = oj + LPR * m;
                if (orow && jo < cnt) {
                    const float xv = __half2float(__ushort_as_half((unsigned short)xraw[m]));
                    float w0, w1;
                    if (!a.w8) {
                        w0 = __half2float(__ushort_as_half((unsigned short)(wraw[m] & 0xffffu)));
                        w1 = __half2float(__ushort_as_half((unsigned short)(wraw[m] >> 16)));
                    } else {
                        w0 = w16_value<__half>(a, kidx[m], nA);
                        w1 = w16_value<__half>(a, kidx[m], nA + 1);
                    }
                    f0 = fmaf(xv, w0, f0);
                    f1 = fmaf(xv, w1, f1);
                }
            }
            // past the registers: through L2, kChainBatch positions per round so that
            // their loads are in flight together (same summation order as one by one)
            for (int jb = oj + LPR * kChainPre; jb < cnt; jb += kChainBatch * LPR) {
                if (!orow) continue;
                int kb[kChainBatch];
                uint32_t xb[kChainBatch], wb[kChainBatch];
#pragma unroll
                for (int u = 0; u < kChainBatch; ++u) {
                    const int jo = jb + u * LPR;
                    kb[u] = jo < cnt ? outlier_col(jo) : 0;
                }
#pragma unroll
                for (int u = 0; u < kChainBatch; ++u) {
                    const int jo = jb + u * LPR;
                    xb[u] = jo < cnt ? outlier_x(oi, jo, kb[u]) : 0u;
                    wb[u] = (jo < cnt && !a.w8) ? chain_ldg_nc_u32(a.W16 + (size_t)kb[u] * N + nA) : 0u;
                }
#pragma unroll
                for (int u = 0; u < kChainBatch; ++u) {
                    if (jb + u * LPR >= cnt) break;
                    const float xv = __half2float(__ushort_as_half((unsigned short)xb[u]));
                    float w0, w1;
                    if (!a.w8) {
                        w0 = __half2float(__ushort_as_half((unsigned short)(wb[u] & 0xffffu)));
                        w1 = __half2float(__ushort_as_half((unsigned short)(wb[u] >> 16)));
                    } else {
                        w0 = w16_value<__half>(a, kb[u], nA);
                        w1 = w16_value<__half>(a, kb[u], nA + 1);
                    }
                    f0 = fmaf(xv, w0, f0);
                    f1 = fmaf(xv, w1, f1);
                }
            }
#pragma unroll
            for (int o = LPR / 2; o >= 1; o >>= 1) {
                f0 += __shfl_xor_sync(0xffffffffu, f0, o);
                f1 += __shfl_xor_sync(0xffffffffu, f1, o);
            }
        }
        // A5
        const bool mine = oj == 0 && orow;
        float y0f = 0.0f, y1f = 0.0f;
        if (mine) {
            const float k2 = 1.0f / 16129.0f;
            const __half y0 = __float2half_rn(fmaf((float)c0, rs * cs0 * k2, f0));
            const __half y1 = __float2half_rn(fmaf((float)c1, rs * cs1 * k2, f1));
            *reinterpret_cast<__half2*>(reinterpret_cast<__half*>(a.out) + (size_t)oi * N + nA) = __halves2half2(y0, y1);
            if (ch.c_out != nullptr) *reinterpret_cast<int2*>(ch.c_out + (size_t)oi * N + nA) = make_int2(c0, c1);
            y0f = fabsf(__half2float(y0));
            y1f = fabsf(__half2float(y1));
        }
        if (EMIT) {
            // the next layer's A1 on these two columns of Y (all rows are here) ...
            const bool o0 = __ballot_sync(0xffffffffu, mine && y0f > ch.next_t) != 0u;
            const bool o1 = __ballot_sync(0xffffffffu, mine && y1f > ch.next_t) != 0u;
            if (lane == 0)
                *reinterpret_cast<uint16_t*>(ch.out + chain_flags_off() + nA) =
                    (uint16_t)((o0 ? 1u : 0u) | (o1 ? 256u : 0u));
            // ... and its row absmax over the non-outlier columns, per strip
            const int pb = j & 1;
            if (j >= 2 && !wait_warp(&sb->strip_free[pb], ((j >> 1) - 1) & 1u, 24)) return;
            if (mine) s_part[pb][warp][oi] = fmaxf(o0 ? 0.0f : y0f, o1 ? 0.0f : y1f);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sb->strip_done[pb]);
            if (warp == 0) {
                if (!wait_warp(&sb->strip_done[pb], (j >> 1) & 1u, 25)) return;
                if (lane < MR) {
                    float m = s_part[pb][0][lane];
                    for (int w = 1; w < kChainWarps; ++w) m = fmaxf(m, s_part[pb][w][lane]);
                    parts_out[(size_t)strip * MR + lane] = m;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sb->strip_free[pb]);
            }
        }
    }
}

}  // namespace llmint8
