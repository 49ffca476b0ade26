// Decode path (M <= 16) of the LLM.int8() matmul: steps A3-A5 in one kernel.
//
// Decode is bound by streaming the int8 weight codes from HBM once (every
// decode step reads all weights: INT8-vs-FP8 page, section 1).  B300's int8
// tensor path is slow (mma.sync s8 and dp4a both top out near 140 TOPS, short
// of the ~110 T MAC/s that 16 rows at full HBM rate need), so the codes are
// widened to exact fp16 integers in registers and multiplied with the legacy
// fp16 MMA (m16n8k16, fp32 accumulate, ~570 TFLOPS).  Every product is an
// integer of magnitude <= 127^2 and every partial sum over <= 1024 products
// stays below 2^24, where fp32 holds integers exactly; after each 1024-long
// K-chunk the fp32 accumulators are converted to int32 and added, so the
// integer result C is exact for any K.
//
// Work split: one CTA per 16 output columns; its 8 warps split K; their int32
// partials are summed in shared memory; the CTA then adds the fp16 outlier
// slice (A4) and applies the scale outer product (A5) -- no global atomics and
// no second kernel.
#pragma once

#include "common.cuh"

namespace llmint8 {

constexpr int kGemvWarps = 8;
constexpr int kGemvCols = 16;

struct GemvArgs {
    const __half* codes;        // [M, K] fp16 code values of X
    const int8_t* Wq;           // [N, K]
    const float* col_scale;     // [N]
    const float* row_scale;     // [M]
    const __half* X;            // [M, K] original activations (outlier values)
    const __half* W16;          // [K, N] retained fp16 weight (outlier rows)
    const WsHeader* hdr;        // outlier_count
    const int32_t* outlier_idx; // [count]
    void* out;                  // Y fp16 [M, N] or C int32 [M, N]
    int M, K, N;
    int k_per_warp;             // multiple of 64
    int use_outliers;           // 0 when the threshold is +inf
};

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// MT = number of 8-row tiles of X (1 for M <= 8, 2 for M <= 16).
//
// Fragment mapping (K is permuted consistently on both operands, which leaves
// the sum unchanged): thread (g = lane/4, t = lane%4) loads 16 contiguous
// bytes of weight rows n0+g and n0+g+8 at k = kb + 16t; MMA j (0..3) takes
// bytes 4j..4j+3 of them, and the matching 4 fp16 codes of X rows g (+8).
template <int MT, bool WRITE_I32>
__global__ void __launch_bounds__(kGemvWarps * 32) k_gemv_decode(GemvArgs a) {
    __shared__ int32_t s_red[kGemvWarps][kGemvCols][16];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, tq = lane & 3;
    const int n0 = blockIdx.x * kGemvCols;
    const int K = a.K;
    const int kb0 = warp * a.k_per_warp;
    const int kend = min(K, kb0 + a.k_per_warp);
    const int nsteps = kend > kb0 ? (kend - kb0 + 63) >> 6 : 0;

    const int8_t* w0p = a.Wq + (size_t)(n0 + g) * K + kb0 + 16 * tq;
    const int8_t* w1p = a.Wq + (size_t)(n0 + g + 8) * K + kb0 + 16 * tq;
    const __half* xp[MT];
    bool xok[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        const int i = g + 8 * t;
        xok[t] = i < a.M;
        xp[t] = a.codes + (size_t)(xok[t] ? i : 0) * K + kb0 + 16 * tq;
    }

    float acc[MT][4];
    int iacc[MT][4];
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            acc[t][r] = 0.0f;
            iacc[t][r] = 0;
        }

    constexpr int D = 4;  // weight prefetch depth (steps of 64 K)
    uint4 wa[D], wb[D];
    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int d = 0; d < D; ++d) {
        const bool ok = d < nsteps && kb0 + d * 64 + 16 * tq < kend;
        wa[d] = ok ? ldg_stream_v4(w0p + d * 64) : z;
        wb[d] = ok ? ldg_stream_v4(w1p + d * 64) : z;
    }

    for (int s0 = 0; s0 < nsteps; s0 += D) {
#pragma unroll
        for (int d = 0; d < D; ++d) {
            const int s = s0 + d;
            if (s < nsteps) {
                const uint4 w0 = wa[d], w1 = wb[d];
                {
                    const int sn = s + D;
                    const bool ok = sn < nsteps && kb0 + sn * 64 + 16 * tq < kend;
                    wa[d] = ok ? ldg_stream_v4(w0p + sn * 64) : z;
                    wb[d] = ok ? ldg_stream_v4(w1p + sn * 64) : z;
                }
                const bool kok = kb0 + s * 64 + 16 * tq < kend;
                uint4 xf[MT][2];
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    const bool ok = xok[t] && kok;
                    xf[t][0] = ok ? ldg_nc_v4(xp[t] + s * 64) : z;
                    xf[t][1] = ok ? ldg_nc_v4(xp[t] + s * 64 + 8) : z;
                }
                const uint32_t wr0[4] = {w0.x, w0.y, w0.z, w0.w};
                const uint32_t wr1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t a0, a2, a1, a3;
                    s8x4_to_half2x2(wr0[j], a0, a2);
                    s8x4_to_half2x2(wr1[j], a1, a3);
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        const uint4& xa = (j < 2) ? xf[t][0] : xf[t][1];
                        const uint32_t b0 = (j & 1) ? xa.z : xa.x;
                        const uint32_t b1 = (j & 1) ? xa.w : xa.y;
                        mma_16816(acc[t], a0, a1, a2, a3, b0, b1);
                    }
                }
                if ((s & 15) == 15) {  // 1024 K done: move the exact partial to int32
#pragma unroll
                    for (int t = 0; t < MT; ++t)
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            iacc[t][r] += __float2int_rn(acc[t][r]);
                            acc[t][r] = 0.0f;
                        }
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int r = 0; r < 4; ++r) iacc[t][r] += __float2int_rn(acc[t][r]);

    // accumulator layout: d0,d1 -> (col g, rows 8t+2tq, +1); d2,d3 -> (col g+8, same rows)
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        const int i0 = 8 * t + 2 * tq;
        s_red[warp][g][i0] = iacc[t][0];
        s_red[warp][g][i0 + 1] = iacc[t][1];
        s_red[warp][g + 8][i0] = iacc[t][2];
        s_red[warp][g + 8][i0 + 1] = iacc[t][3];
    }
    __syncthreads();

    const int nl = threadIdx.x & 15, i = threadIdx.x >> 4;
    if (i >= a.M) return;
    const int n = n0 + nl;
    int32_t c = 0;
#pragma unroll
    for (int w = 0; w < kGemvWarps; ++w) c += s_red[w][nl][i];
    if (WRITE_I32) {
        reinterpret_cast<int32_t*>(a.out)[(size_t)i * a.N + n] = c;
        return;
    }
    float f = 0.0f;
    if (a.use_outliers) {
        const int cnt = a.hdr->outlier_count;
        const __half* xr = a.X + (size_t)i * K;
        for (int j = 0; j < cnt; ++j) {
            const int k = a.outlier_idx[j];
            f = fmaf(__half2float(xr[k]), __half2float(a.W16[(size_t)k * a.N + n]), f);
        }
    }
    const float scale = a.row_scale[i] * a.col_scale[n] * (1.0f / 16129.0f);
    reinterpret_cast<__half*>(a.out)[(size_t)i * a.N + n] = __float2half_rn(fmaf((float)c, scale, f));
}

}  // namespace llmint8
