// Decode path (M <= 16) of the LLM.int8() matmul: steps A3-A5 in one kernel.
//
// Decode is bound by streaming the int8 weight codes from HBM once (every
// decode step reads all weights: INT8-vs-FP8 page, section 1).  The product
// uses the int8 mma.sync (m16n8k32, s8 x s8 -> s32): it consumes the weight
// bytes as they arrive, with no widening, and accumulates exactly in int32
// (A3).  Its ~140 TOPS on B300 covers 8 activation rows at full HBM rate; at
// 16 rows it is the limit near 70 % of the HBM roofline.
//
// Streaming: one CTA per 16 output columns, K split over 8 warps.  Each warp
// keeps gemv_ring(MT) steps in flight through a private shared-memory ring
// filled with cp.async.  A ring slot holds one step of both operands: 1 KB of
// weights (16 rows x 64 K) and the matching 16-byte fragments of the X codes
// (64 K x up to 16 rows), so the codes, which sit in L2, get the same
// lookahead as the weights: an L2 hit takes over a microsecond while HBM
// streams at full rate, far longer than a few steps of compute.  Each thread
// copies, and later reads back, its own bytes of a slot, so the ring needs no
// cross-thread synchronization.  The weight halves of the first slots are
// requested before griddepcontrol.wait (weights do not depend on the X pass),
// so they overlap the X pass under programmatic dependent launch; the code
// halves follow right after the wait.
//
// Epilogue: the 8 warps' int32 partials are summed in shared memory (each
// warp's drained ring); the CTA adds the fp16 outlier slice (A4, fp32
// accumulation, operands staged in shared memory while the weights stream) and
// applies the scale outer product (A5).  Everything the epilogue reads from
// global memory is requested at kernel start.
#pragma once

#include "common.cuh"
#include "xpass.cuh"

namespace llmint8 {

constexpr int kGemvWarps = 8;
constexpr int kGemvCols = 16;
constexpr int kGemvOutChunk = 128;  // outlier columns staged in shared memory at a time

// Ring of one warp: steps in flight, and bytes per step for M rows of X: 1 KB of
// weights plus 64 bytes of X codes per row (the 4 threads of a row hold 16
// bytes each).  The ring takes at most 96 KB per CTA, so two CTAs fit on an SM
// next to the static staging buffers; 8 steps cover a whole K = 4096 slice.
__host__ __device__ constexpr int gemv_ring(int mt) { return mt == 1 ? 8 : 6; }
__host__ __device__ constexpr int gemv_slot(int M) { return 1024 + 64 * M; }
__host__ __device__ constexpr size_t gemv_dyn_smem(int M) {
    return (size_t)kGemvWarps * gemv_ring(M <= 8 ? 1 : 2) * gemv_slot(M);
}

struct GemvArgs {
    const int8_t* codes;        // [M, K] int8 codes of X
    const int8_t* Wq;           // [N, K]
    const float* col_scale;     // [N]
    const float* row_scale;     // [M]
    const __half* W16;          // [K, N] retained fp16 weight (outlier rows)
    const WsHeader* hdr;        // outlier_count
    const int32_t* outlier_idx; // [count]
    const __half* xo;           // [M, xo_pitch] outlier columns of X, zero-padded to a multiple of 64
    int xo_pitch;
    void* out;                  // Y fp16 [M, N] or C int32 [M, N]
    int M, K, N;
    int k_per_warp;             // multiple of 64
    int use_outliers;           // 0 when the threshold is +inf
    // w8 = 1: no full fp16 copy of W (W16 unused).  Row k of W for the outlier
    // slice is W16c[row_map[k]] when 0 <= row_map[k] < w16_rows, else the
    // dequantized codes Wq[., k] with the column scales.
    int w8;
    const __half* W16c;         // [w16_rows, N] kept fp16 rows of W
    const int32_t* row_map;     // [K] (nullptr: no row kept)
    int w16_rows;
};

// Columns nb .. nb+7 of row k of W (the A4 operand) into 16 bytes of shared
// memory: by cp.async from the fp16 copy or a kept row, or dequantized from the
// codes.  The codes are requested here into registers (their loads stay in
// flight while the weights stream) and converted by w8_finish before the
// staged rows are read.  All sources are constant inputs.
struct W8Pending {
    int q[8];
    __half* dst;  // nullptr: nothing pending
    int nb;
};

__device__ __forceinline__ int ldg_nc_s8(const int8_t* p) {
    int v;
    asm volatile("ld.global.nc.s8 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

template <typename T>
__device__ __forceinline__ void stage_w16_8(const GemvArgs& a, __half* dst, int k, int nb, W8Pending& pend) {
    if (!a.w8) {
        cp_async16(dst, a.W16 + (size_t)k * a.N + nb);
        return;
    }
    const int rm = a.row_map != nullptr ? __ldg(a.row_map + k) : -1;
    if (rm >= 0 && rm < a.w16_rows) {
        cp_async16(dst, a.W16c + (size_t)rm * a.N + nb);
        return;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) pend.q[e] = ldg_nc_s8(a.Wq + (size_t)(nb + e) * a.K + k);
    pend.dst = dst;
    pend.nb = nb;
}

template <typename T>
__device__ __forceinline__ void w8_finish(const GemvArgs& a, W8Pending& pend) {
    if (pend.dst == nullptr) return;
    uint32_t h[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __half lo = dequant_weight<T>((int8_t)pend.q[2 * e], a.col_scale[pend.nb + 2 * e]);
        const __half hi = dequant_weight<T>((int8_t)pend.q[2 * e + 1], a.col_scale[pend.nb + 2 * e + 1]);
        h[e] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
    }
    *reinterpret_cast<uint4*>(pend.dst) = make_uint4(h[0], h[1], h[2], h[3]);
    pend.dst = nullptr;
}

// One element of row k of W (the A4 operand) at column n, from the same sources.
template <typename T>
__device__ __forceinline__ float w16_value(const GemvArgs& a, int k, int n) {
    if (!a.w8) return elem_f<T>(a.W16[(size_t)k * a.N + n]);
    const int rm = a.row_map != nullptr ? __ldg(a.row_map + k) : -1;
    if (rm >= 0 && rm < a.w16_rows) return elem_f<T>(a.W16c[(size_t)rm * a.N + n]);
    return elem_f<T>(dequant_weight<T>(a.Wq[(size_t)n * a.K + k], a.col_scale[n]));
}

__device__ __forceinline__ void imma_16832(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// MT = number of 8-row tiles of X (1 for M <= 8, 2 for M <= 16).
//
// Fragment mapping.  The MMA's rows are 16 weight rows (output columns n0..n0+15),
// its columns are 8 rows of X, and K is permuted consistently on both operands
// (which leaves every dot product unchanged): thread (g = lane/4, q = lane%4)
// holds 16 contiguous bytes of weight rows n0+g and n0+g+8 at k = kb + 16q, and
// 16 bytes of X row g (+8) at the same k.  MMA j (0, 1) takes bytes 8j..8j+7 of
// each: the first word as the k-slot 4q..4q+3 fragment, the second as 16+4q..
//
// Ring slot of step s (thread-private bytes at lane * 16):
//   [0, 512) weight row n0+g, [512, 1024) weight row n0+g+8,
//   [1024 + 512 t, ...) X codes of row g + 8t (only rows < M are copied and
//   read, so the slot is 1024 + 64 M bytes).
// Commit groups: one per weight step before the wait (R), the X halves of those
// R steps (one group), the outlier staging (one group), then one group per
// refilled step.
template <int MT, bool WRITE_I32, typename T>
__global__ void __launch_bounds__(kGemvWarps * 32, 2) k_gemv_decode(GemvArgs a) {
    constexpr int R = gemv_ring(MT);
    const int SLOT = gemv_slot(a.M);
    __shared__ __align__(16) __half s_w16o[kGemvOutChunk][kGemvCols];  // W16[O[j], n0..n0+15]
    __shared__ __align__(16) __half s_xo[16][kGemvOutChunk];           // X[i, O[j]]
    extern __shared__ __align__(16) uint8_t s_ring_all[];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tq = lane & 3;
    const int n0 = blockIdx.x * kGemvCols;
    const int K = a.K;
    const int kb0 = warp * a.k_per_warp;
    const int kend = min(K, kb0 + a.k_per_warp);
    const int nsteps = kend > kb0 ? (kend - kb0 + 63) >> 6 : 0;

    const int8_t* w0p = a.Wq + (size_t)(n0 + g) * K + kb0 + 16 * tq;
    const int8_t* w1p = a.Wq + (size_t)(n0 + g + 8) * K + kb0 + 16 * tq;
    const int8_t* xp[MT];
    bool xok[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        const int i = g + 8 * t;
        xok[t] = i < a.M;
        xp[t] = a.codes + (size_t)(xok[t] ? i : 0) * K + kb0 + 16 * tq;
    }
    uint8_t* ring = s_ring_all + (size_t)warp * R * SLOT;
    auto slot_of = [&](int sn) { return ring + (sn % R) * SLOT + lane * 16; };
    auto step_ok = [&](int sn) { return sn < nsteps && kb0 + sn * 64 + 16 * tq < kend; };
    auto issue_w = [&](int sn) {
        if (step_ok(sn)) {
            uint8_t* slot = slot_of(sn);
            cp_async16(slot, w0p + sn * 64);
            cp_async16(slot + 512, w1p + sn * 64);
        }
    };
    auto issue_x = [&](int sn) {
        if (step_ok(sn)) {
            uint8_t* slot = slot_of(sn);
#pragma unroll
            for (int t = 0; t < MT; ++t)
                if (xok[t]) cp_async16(slot + 1024 + 512 * t, xp[t] + sn * 64);
        }
    };

    // epilogue thread mapping: (row ri, column n0 + nl)
    const int nl = tid & 15, ri = tid >> 4;
    const bool active = ri < a.M;
    const int n = n0 + nl;
    // constant inputs may be read before the wait
    const float cs = WRITE_I32 ? 0.0f : a.col_scale[n];
    pdl_trigger();
#pragma unroll
    for (int d = 0; d < R; ++d) {
        issue_w(d);
        cp_async_commit();
    }
    pdl_wait();
#pragma unroll
    for (int d = 0; d < R; ++d) issue_x(d);
    cp_async_commit();
    const float rs = (!WRITE_I32 && active) ? __ldcg(a.row_scale + ri) : 0.0f;

    // A4 operands of this CTA's 16 columns for outlier positions [base, base + c):
    // the W16 rows (32 bytes each) and the gathered X values.  The indices of the
    // first chunk are requested together with the count (positions past it are
    // loaded but not used), so the W16 gather waits for one L2 round trip.
    static_assert(2 * kGemvOutChunk <= kGemvWarps * 32, "one (outlier, half-row) per thread");
    const bool outl = !WRITE_I32 && a.use_outliers;
    const int nidx = min(K, kGemvOutChunk);
    const int k_first = (outl && (tid >> 1) < nidx) ? ldg_cg_s32(a.outlier_idx + (tid >> 1)) : 0;
    const int cnt = outl ? ldg_cg_s32(&a.hdr->outlier_count) : 0;
    W8Pending pend;
    pend.dst = nullptr;
    auto stage_outliers = [&](int base, int c) {
        for (int e = tid; e < 2 * nidx; e += kGemvWarps * 32) {
            const int j = e >> 1, hv = e & 1;
            const int k = base == 0 ? k_first : (base + j < K ? __ldcg(a.outlier_idx + base + j) : 0);
            if (j < c) stage_w16_8<T>(a, &s_w16o[j][hv * 8], k, n0 + hv * 8, pend);
        }
        const int cv = (c + 7) >> 3;
        for (int e = tid; e < a.M * (kGemvOutChunk / 8); e += kGemvWarps * 32) {
            const int i = e / (kGemvOutChunk / 8), qv = e - i * (kGemvOutChunk / 8);
            if (qv < cv) cp_async16(&s_xo[i][qv * 8], a.xo + (size_t)i * a.xo_pitch + base + qv * 8);
        }
        cp_async_commit();
    };
    if (cnt > 0)
        stage_outliers(0, min(cnt, kGemvOutChunk));
    else
        cp_async_commit();  // keep the group count fixed

    int acc[MT][4];
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[t][r] = 0;
    // Main loop, unrolled by the ring depth: ring offsets and the offsets of the
    // refill sources are constants, the sources advance by R steps per round.
    // Steps [0, nfull) are whole 64-byte steps inside the warp's K slice; only a
    // ragged last step (K not a multiple of 64) takes the checked path.
    const uint4 z = make_uint4(0, 0, 0, 0);
    const int nfull = kend > kb0 ? (kend - kb0) >> 6 : 0;
    uint8_t* const my_ring = ring + lane * 16;
    const int8_t* wr = w0p + R * 64;  // refill source of step R: row n0+g; row n0+g+8 is 8K further
    const int8_t* xr[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) xr[t] = xp[t] + R * 64;
    for (int base = 0; base < nsteps; base += R) {
#pragma unroll
        for (int d = 0; d < R; ++d) {
            const int s = base + d;
            if (s >= nsteps) break;
            if (base > 0)
                cp_async_wait_group<R - 1>();  // the refill of step s was committed R - 1 groups ago
            else if (d == 0)
                cp_async_wait_group<1>();      // the first R steps, both halves (staging may be pending)
            uint8_t* slot = my_ring + d * SLOT;
            const uint4 w0 = *reinterpret_cast<const uint4*>(slot);
            const uint4 w1 = *reinterpret_cast<const uint4*>(slot + 512);
            const bool ok = s < nfull || kb0 + s * 64 + 16 * tq < kend;
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const uint4 xf = (ok && xok[t]) ? *reinterpret_cast<const uint4*>(slot + 1024 + 512 * t) : z;
                imma_16832(acc[t], w0.x, w1.x, w0.y, w1.y, xf.x, xf.y);
                imma_16832(acc[t], w0.z, w1.z, w0.w, w1.w, xf.z, xf.w);
            }
            // the slot's values were consumed by the MMAs above: refill it with step s + R
            const int sr = s + R;
            if (sr < nfull || (sr < nsteps && kb0 + sr * 64 + 16 * tq < kend)) {
                cp_async16(slot, wr + d * 64);
                cp_async16(slot + 512, wr + (size_t)8 * K + d * 64);
#pragma unroll
                for (int t = 0; t < MT; ++t)
                    if (xok[t]) cp_async16(slot + 1024 + 512 * t, xr[t] + d * 64);
            }
            cp_async_commit();
        }
        wr += R * 64;
#pragma unroll
        for (int t = 0; t < MT; ++t) xr[t] += R * 64;
    }

    // No copy may still target shared memory: the ring is drained (its later
    // groups are empty) and the staging group has landed.  Each warp's partials
    // then go to its own ring, [16 x rows][16 columns] int32.
    w8_finish<T>(a, pend);
    cp_async_wait_all();
    int32_t* red = reinterpret_cast<int32_t*>(ring);
    // accumulator layout: d0,d1 -> (column g, x rows 8t+2q, +1); d2,d3 -> (column g+8, same rows)
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        const int i0 = 8 * t + 2 * tq;
        red[i0 * kGemvCols + g] = acc[t][0];
        red[(i0 + 1) * kGemvCols + g] = acc[t][1];
        red[i0 * kGemvCols + g + 8] = acc[t][2];
        red[(i0 + 1) * kGemvCols + g + 8] = acc[t][3];
    }
    __syncthreads();

    int32_t c = 0;
    if (active) {
#pragma unroll
        for (int w = 0; w < kGemvWarps; ++w)
            c += reinterpret_cast<const int32_t*>(s_ring_all + (size_t)w * R * SLOT)[ri * kGemvCols + nl];
    }
    if (WRITE_I32) {
        if (active) reinterpret_cast<int32_t*>(a.out)[(size_t)ri * a.N + n] = c;
        return;
    }
    float f = 0.0f;
    if (cnt > 0) {
        for (int base = 0;;) {
            const int cc = min(kGemvOutChunk, cnt - base);
            if (active)
                for (int j = 0; j < cc; ++j) f = fmaf(elem_f<T>(s_xo[ri][j]), elem_f<T>(s_w16o[j][nl]), f);
            base += kGemvOutChunk;
            if (base >= cnt) break;
            __syncthreads();
            stage_outliers(base, min(kGemvOutChunk, cnt - base));
            w8_finish<T>(a, pend);
            cp_async_wait_all();
            __syncthreads();
        }
    }
    if (active) {
        const float scale = rs * cs * (1.0f / 16129.0f);
        reinterpret_cast<uint16_t*>(a.out)[(size_t)ri * a.N + n] = Fmt<T>::from_float(fmaf((float)c, scale, f));
    }
}

// Persistent form for shapes with more 16-column tiles than resident CTAs
// (two per SM), used for up to 8 rows of X.  One-tile CTAs would run in several waves, and every later
// wave would start its weight stream from an empty ring while the SM's share
// of HBM idles.  Here the grid is exactly the resident CTAs; CTA b takes tiles
// b, b + G, b + 2G, ... (G = grid size), and each warp's ring runs on across
// the CTA's tiles, so the next tile's weights stream while the current one is
// reduced and written.  The first ring steps are requested before the
// dependency wait, as in the one-tile kernel.
//
// Tile epilogue, between two CTA barriers: the 8 warps' partials are summed in
// shared memory, the fp16 outlier slice (A4) is added from staged operands and
// the scale outer product applied (A5).  The gathered X values of the first
// kTileOutChunk outliers are staged once; the matching W16 rows of the next
// tile are staged during the current one (double-buffered).  Outliers past the
// first chunk are staged chunk by chunk in the epilogue (their X values into a
// buffer of their own, their W16 rows into the tile's staging buffer once every
// thread has read it).
//
// Commit groups of every thread, in order: one per weight step before the wait
// (R), the X halves of those steps, the staging of tile 0 (X values and W16
// rows), then one per refilled step, and after each tile but the last the W16
// staging of the next tile.
constexpr int kTileOutChunk = 64;

template <int MT, bool WRITE_I32, typename T>
__global__ void __launch_bounds__(kGemvWarps * 32, 2) k_gemv_decode_tiles(GemvArgs a) {
    constexpr int R = gemv_ring(MT);
    constexpr int MR = 8 * MT;  // rows of X held by the fragments
    const int SLOT = gemv_slot(a.M);
    __shared__ int32_t s_red[kGemvWarps][MR][kGemvCols];                   // int8 partials of one tile
    __shared__ __align__(16) __half s_w16o[2][kTileOutChunk][kGemvCols];  // W16[O[j], tile columns]
    __shared__ __align__(16) __half s_xo[MR][kTileOutChunk];              // X[i, O[j]]
    __shared__ __align__(16) __half s_xo2[MR][kTileOutChunk];             // X values of a later chunk
    __shared__ int32_t s_idx[kTileOutChunk];                               // O[j]
    extern __shared__ __align__(16) uint8_t s_ring_all[];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tq = lane & 3;
    const int K = a.K;
    const int kb0 = warp * a.k_per_warp;
    const int kend = min(K, kb0 + a.k_per_warp);
    const int nsteps = kend > kb0 ? (kend - kb0 + 63) >> 6 : 0;
    const int G = gridDim.x;
    const int my_tiles = (a.N / kGemvCols - (int)blockIdx.x + G - 1) / G;  // >= 1: the grid has <= tiles CTAs
    const int total = my_tiles * nsteps;
    auto tile_n0 = [&](int j) { return ((int)blockIdx.x + j * G) * kGemvCols; };

    const int8_t* xp[MT];
    bool xok[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        const int i = g + 8 * t;
        xok[t] = i < a.M;
        xp[t] = a.codes + (size_t)(xok[t] ? i : 0) * K + kb0 + 16 * tq;
    }
    uint8_t* ring = s_ring_all + (size_t)warp * R * SLOT;
    auto slot_of = [&](int u) { return ring + (u % R) * SLOT + lane * 16; };
    auto step_ok = [&](int st) { return st < nsteps && kb0 + st * 64 + 16 * tq < kend; };
    // flattened step u = (tile j of this CTA) * nsteps + (step st of the warp's K slice)
    auto issue_w = [&](int u) {
        if (u < total) {
            const int j = u / nsteps, st = u - j * nsteps;
            if (step_ok(st)) {
                const int8_t* w = a.Wq + (size_t)(tile_n0(j) + g) * K + kb0 + 64 * st + 16 * tq;
                uint8_t* slot = slot_of(u);
                cp_async16(slot, w);
                cp_async16(slot + 512, w + (size_t)8 * K);
            }
        }
    };
    auto issue_x = [&](int u) {
        if (u < total) {
            const int st = u % nsteps;
            if (step_ok(st)) {
                uint8_t* slot = slot_of(u);
#pragma unroll
                for (int t = 0; t < MT; ++t)
                    if (xok[t]) cp_async16(slot + 1024 + 512 * t, xp[t] + 64 * st);
            }
        }
    };

    // epilogue thread mapping: (row ri, tile column nl)
    const int nl = tid & 15, ri = tid >> 4;
    const bool active = ri < a.M;
    // constant inputs may be read before the wait
    float cs_next = WRITE_I32 ? 0.0f : a.col_scale[tile_n0(0) + nl];
    pdl_trigger();
#pragma unroll
    for (int d = 0; d < R; ++d) {
        issue_w(d);
        cp_async_commit();
    }
    pdl_wait();
#pragma unroll
    for (int d = 0; d < R; ++d) issue_x(d);
    cp_async_commit();
    const float rs = (!WRITE_I32 && active) ? __ldcg(a.row_scale + ri) : 0.0f;

    // A4 operands: indices requested together with the count (positions past it
    // are loaded but not used)
    const bool outl = !WRITE_I32 && a.use_outliers;
    const int idx0 = (outl && tid < kTileOutChunk && tid < K) ? ldg_cg_s32(a.outlier_idx + tid) : 0;
    const int cnt = outl ? ldg_cg_s32(&a.hdr->outlier_count) : 0;
    const int cst = min(cnt, kTileOutChunk);
    if (tid < kTileOutChunk) s_idx[tid] = idx0;
    {
        // the gathered X values are zero-padded past the count up to a multiple of 64
        const int cv = (cst + 7) >> 3;
        for (int e = tid; e < a.M * (kTileOutChunk / 8); e += kGemvWarps * 32) {
            const int i = e / (kTileOutChunk / 8), qv = e - i * (kTileOutChunk / 8);
            if (qv < cv) cp_async16(&s_xo[i][qv * 8], a.xo + (size_t)i * a.xo_pitch + qv * 8);
        }
    }
    __syncthreads();  // s_idx
    W8Pending pend;  // dequantized rows of the staged tile, converted before its epilogue
    pend.dst = nullptr;
    auto stage_w16 = [&](int buf, int n0) {
        for (int e = tid; e < 2 * cst; e += kGemvWarps * 32) {
            const int jx = e >> 1, hv = e & 1;
            stage_w16_8<T>(a, &s_w16o[buf][jx][hv * 8], s_idx[jx], n0 + hv * 8, pend);
        }
        cp_async_commit();
    };
    stage_w16(0, tile_n0(0));

    // Refill cursor: the step u + R as (tile jr, step sr of the warp's slice) and
    // its weight source; the ring slot of step u is sl.  Both advance without
    // divisions.  Steps [0, nfull) of a slice are whole 64-byte steps.
    const int nfull = kend > kb0 ? (kend - kb0) >> 6 : 0;
    uint8_t* const my_ring = ring + lane * 16;
    int jr = nsteps > 0 ? R / nsteps : my_tiles, sr = nsteps > 0 ? R % nsteps : 0;
    auto w_src = [&](int jt) { return a.Wq + (size_t)(tile_n0(jt) + g) * K + kb0 + 16 * tq; };
    const int8_t* wr = jr < my_tiles ? w_src(jr) + 64 * sr : nullptr;
    int sl = 0;
    const uint4 z = make_uint4(0, 0, 0, 0);
    int u = 0;
    for (int j = 0; j < my_tiles; ++j) {
        int acc[MT][4];
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[t][r] = 0;
        for (int st = 0; st < nsteps; ++st, ++u) {
            if (u == 0)
                cp_async_wait_group<1>();      // the first R steps, both halves (staging may be pending)
            else if (u >= R)
                cp_async_wait_group<R - 1>();  // at least R - 1 groups followed the refill of step u
            uint8_t* slot = my_ring + sl * SLOT;
            const uint4 w0 = *reinterpret_cast<const uint4*>(slot);
            const uint4 w1 = *reinterpret_cast<const uint4*>(slot + 512);
            const bool ok = st < nfull || kb0 + st * 64 + 16 * tq < kend;
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const uint4 xf = (ok && xok[t]) ? *reinterpret_cast<const uint4*>(slot + 1024 + 512 * t) : z;
                imma_16832(acc[t], w0.x, w1.x, w0.y, w1.y, xf.x, xf.y);
                imma_16832(acc[t], w0.z, w1.z, w0.w, w1.w, xf.z, xf.w);
            }
            // the slot's values were consumed by the MMAs above: refill it with step u + R
            if (jr < my_tiles && (sr < nfull || kb0 + sr * 64 + 16 * tq < kend)) {
                cp_async16(slot, wr);
                cp_async16(slot + 512, wr + (size_t)8 * K);
#pragma unroll
                for (int t = 0; t < MT; ++t)
                    if (xok[t]) cp_async16(slot + 1024 + 512 * t, xp[t] + 64 * sr);
            }
            cp_async_commit();
            wr += 64;
            if (++sr == nsteps) {
                sr = 0;
                if (++jr < my_tiles) wr = w_src(jr);
            }
            sl = sl + 1 == R ? 0 : sl + 1;
        }
        // accumulator layout: d0,d1 -> (column g, x rows 8t+2q, +1); d2,d3 -> (column g+8, same rows)
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            const int i0 = 8 * t + 2 * tq;
            s_red[warp][i0][g] = acc[t][0];
            s_red[warp][i0 + 1][g] = acc[t][1];
            s_red[warp][i0][g + 8] = acc[t][2];
            s_red[warp][i0 + 1][g + 8] = acc[t][3];
        }
        const float cs = cs_next;
        if (!WRITE_I32 && j + 1 < my_tiles) cs_next = a.col_scale[tile_n0(j + 1) + nl];
        // this tile's staging has landed once at most R - 1 groups are pending:
        // the nsteps refill groups of the tile followed it
        if (nsteps >= R - 1)
            cp_async_wait_group<R - 1>();
        else
            cp_async_wait_all();
        w8_finish<T>(a, pend);
        __syncthreads();  // partials and staged operands visible to all
        // the other staging buffer was last read by the previous tile's
        // epilogue, which every thread finished before the barrier ending it
        if (j + 1 < my_tiles) stage_w16((j + 1) & 1, tile_n0(j + 1));

        const int n = tile_n0(j) + nl;
        int32_t c = 0;
        if (active) {
#pragma unroll
            for (int w = 0; w < kGemvWarps; ++w) c += s_red[w][ri][nl];
        }
        if (WRITE_I32) {
            if (active) reinterpret_cast<int32_t*>(a.out)[(size_t)ri * a.N + n] = c;
        } else {
            float f = 0.0f;
            if (active)
                for (int jj = 0; jj < cst; ++jj)
                    f = fmaf(elem_f<T>(s_xo[ri][jj]), elem_f<T>(s_w16o[j & 1][jj][nl]), f);
            // past the first chunk: each further chunk is staged by all threads (the
            // count is the same for every thread, so every thread meets the barriers)
            for (int base = cst; base < cnt; base += kTileOutChunk) {
                const int c2 = min(kTileOutChunk, cnt - base);
                W8Pending pend2;  // the next tile's staging may have its own pending rows
                pend2.dst = nullptr;
                __syncthreads();  // the staging buffer and s_xo2 have been read
                for (int e = tid; e < 2 * c2; e += kGemvWarps * 32) {
                    const int jx = e >> 1, hv = e & 1;
                    stage_w16_8<T>(a, &s_w16o[j & 1][jx][hv * 8], ldg_cg_s32(a.outlier_idx + base + jx),
                                   tile_n0(j) + hv * 8, pend2);
                }
                const int cv = (c2 + 7) >> 3;  // the gathered X values are zero-padded past the count
                for (int e = tid; e < a.M * (kTileOutChunk / 8); e += kGemvWarps * 32) {
                    const int i = e / (kTileOutChunk / 8), qv = e - i * (kTileOutChunk / 8);
                    if (qv < cv) cp_async16(&s_xo2[i][qv * 8], a.xo + (size_t)i * a.xo_pitch + base + qv * 8);
                }
                cp_async_commit();
                cp_async_wait_all();
                w8_finish<T>(a, pend2);
                __syncthreads();
                if (active)
                    for (int jj = 0; jj < c2; ++jj)
                        f = fmaf(elem_f<T>(s_xo2[ri][jj]), elem_f<T>(s_w16o[j & 1][jj][nl]), f);
            }
            if (active) {
                const float scale = rs * cs * (1.0f / 16129.0f);
                reinterpret_cast<uint16_t*>(a.out)[(size_t)ri * a.N + n] =
                    Fmt<T>::from_float(fmaf((float)c, scale, f));
            }
        }
        __syncthreads();  // s_red and this tile's staging buffer may be overwritten
    }
    cp_async_wait_all();  // no copy may still target shared memory when the CTA ends
}

}  // namespace llmint8
