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
// keeps kGemvRing steps of 1 KB (16 weight rows x 64 K) in flight through a
// private shared-memory ring filled with cp.async; each thread copies, and
// later reads back, its own 32 bytes of a step, so the ring needs no
// cross-thread synchronization.  With two CTAs per SM that is ~128 KB per SM:
// most of the matrix of the smaller decode shapes is requested at kernel start.
// The copies are issued before griddepcontrol.wait (the weights do not depend
// on the X pass), so they overlap the X pass when launched with programmatic
// dependent launch.
//
// Epilogue: the 8 warps' int32 partials are summed in shared memory; the CTA
// adds the fp16 outlier slice (A4, fp32 accumulation, operands prefetched to
// shared memory) and applies the scale outer product (A5).
#pragma once

#include "common.cuh"
#include "xpass.cuh"

namespace llmint8 {

constexpr int kGemvWarps = 8;
constexpr int kGemvCols = 16;
constexpr int kGemvOutChunk = 256;  // outlier columns staged in shared memory at a time
constexpr int kGemvRing = 8;        // weight steps in flight per warp (1 KB each)
constexpr size_t kGemvDynSmem = (size_t)kGemvWarps * kGemvRing * 1024;

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
};

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
template <int MT, bool WRITE_I32>
__global__ void __launch_bounds__(kGemvWarps * 32, 2) k_gemv_decode(GemvArgs a) {
    __shared__ int32_t s_red[kGemvWarps][16][kGemvCols];                // [warp][x row][column]
    __shared__ __align__(16) __half s_w16o[kGemvOutChunk][kGemvCols];  // W16[O[j], n0..n0+15]
    __shared__ __align__(16) __half s_xo[16][kGemvOutChunk];           // X[i, O[j]]
    extern __shared__ __align__(16) uint8_t s_ring_all[];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
    int acc[MT][4];
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[t][r] = 0;

    uint8_t* ring = s_ring_all + (size_t)warp * kGemvRing * 1024;
    const uint4 z = make_uint4(0, 0, 0, 0);
    auto step_ok = [&](int sn) { return sn < nsteps && kb0 + sn * 64 + 16 * tq < kend; };
    auto issue_w = [&](int sn) {  // one commit group per step, empty past the end
        if (step_ok(sn)) {
            uint8_t* slot = ring + (sn % kGemvRing) * 1024 + lane * 16;
            cp_async16(slot, w0p + sn * 64);
            cp_async16(slot + 512, w1p + sn * 64);
        }
        cp_async_commit();
    };
    constexpr int DX = 4;  // X fragments in flight (steps)
    uint4 xr[DX][MT];
    auto load_x = [&](int sn, uint4 (&x)[MT]) {
        const bool ok = step_ok(sn);
#pragma unroll
        for (int t = 0; t < MT; ++t) x[t] = (ok && xok[t]) ? ldg_cg_v4(xp[t] + sn * 64) : z;
    };

    // Weights are constant inputs: request them before waiting for the X pass,
    // whose codes, scales and outlier list are read only after pdl_wait().
    pdl_trigger();
#pragma unroll
    for (int d = 0; d < kGemvRing; ++d) issue_w(d);
    pdl_wait();
#pragma unroll
    for (int d = 0; d < DX; ++d) load_x(d, xr[d]);

    // A4 operands of this CTA's 16 columns, copied to shared memory while the
    // weights stream: the outlier rows of W16 (32 bytes each) and the gathered
    // outlier values of X (one more commit group).
    const int cnt = (!WRITE_I32 && a.use_outliers) ? __ldcg(&a.hdr->outlier_count) : 0;
    auto stage_outliers = [&](int base, int c) {
        for (int e = threadIdx.x; e < 2 * c; e += kGemvWarps * 32) {
            const int j = e >> 1, hv = e & 1;
            const int k = __ldcg(a.outlier_idx + base + j);
            cp_async16(&s_w16o[j][hv * 8], a.W16 + (size_t)k * a.N + n0 + hv * 8);
        }
        const int cv = (c + 7) >> 3;
        for (int e = threadIdx.x; e < a.M * cv; e += kGemvWarps * 32) {
            const int i = e / cv, qv = e - i * cv;
            cp_async16(&s_xo[i][qv * 8], a.xo + (size_t)i * a.xo_pitch + base + qv * 8);
        }
        cp_async_commit();
    };
    if (cnt > 0) stage_outliers(0, min(cnt, kGemvOutChunk));

    for (int s0 = 0; s0 < nsteps; s0 += DX) {
#pragma unroll
        for (int d = 0; d < DX; ++d) {
            const int s = s0 + d;
            if (s < nsteps) {
                // every group older than the newest kGemvRing-1 is complete: step s has landed
                cp_async_wait_group<kGemvRing - 1>();
                const uint8_t* slot = ring + (s % kGemvRing) * 1024 + lane * 16;
                const uint4 w0 = *reinterpret_cast<const uint4*>(slot);
                const uint4 w1 = *reinterpret_cast<const uint4*>(slot + 512);
                uint4 xf[MT];
#pragma unroll
                for (int t = 0; t < MT; ++t) xf[t] = xr[d][t];
                load_x(s + DX, xr[d]);
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    imma_16832(acc[t], w0.x, w1.x, w0.y, w1.y, xf[t].x, xf[t].y);
                    imma_16832(acc[t], w0.z, w1.z, w0.w, w1.w, xf[t].z, xf[t].w);
                }
                // the slot's values were consumed by the MMAs above: refill it
                issue_w(s + kGemvRing);
            }
        }
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
    __syncthreads();

    const int nl = threadIdx.x & 15, i = threadIdx.x >> 4;
    const bool active = i < a.M;
    const int n = n0 + nl;
    int32_t c = 0;
    if (active) {
#pragma unroll
        for (int w = 0; w < kGemvWarps; ++w) c += s_red[w][i][nl];
    }
    cp_async_wait_all();  // no copy may still target shared memory when the CTA ends
    if (WRITE_I32) {
        if (active) reinterpret_cast<int32_t*>(a.out)[(size_t)i * a.N + n] = c;
        return;
    }
    float f = 0.0f;
    if (cnt > 0) {
        __syncthreads();
        for (int base = 0;;) {
            const int cc = min(kGemvOutChunk, cnt - base);
            if (active)
                for (int j = 0; j < cc; ++j) f = fmaf(__half2float(s_xo[i][j]), __half2float(s_w16o[j][nl]), f);
            base += kGemvOutChunk;
            if (base >= cnt) break;
            __syncthreads();
            stage_outliers(base, min(kGemvOutChunk, cnt - base));
            cp_async_wait_all();
            __syncthreads();
        }
    }
    if (active) {
        const float scale = __ldcg(a.row_scale + i) * a.col_scale[n] * (1.0f / 16129.0f);
        reinterpret_cast<__half*>(a.out)[(size_t)i * a.N + n] = __float2half_rn(fmaf((float)c, scale, f));
    }
}

}  // namespace llmint8
