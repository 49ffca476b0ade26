// Operands of the decode GEMVs (the streaming kernel in gemv_stream.cuh and the
// decode chain in chain.cuh) and the helpers they share: the outlier slice's
// weight source and the int8 mma.sync.
#pragma once

#include "common.cuh"
#include "xpass.cuh"

namespace llmint8 {

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
    int use_outliers;           // 0 when the threshold is +inf
    // w8 = 1: no full fp16 copy of W (W16 unused).  Row k of W for the outlier
    // slice is W16c[row_map[k]] when 0 <= row_map[k] < w16_rows, else the
    // dequantized codes Wq[., k] with the column scales.
    int w8;
    const __half* W16c;         // [w16_rows, N] kept fp16 rows of W
    const int32_t* row_map;     // [K] (nullptr: no row kept)
    int w16_rows;
    WsHeader* hdr_err;          // error word (bounded waits of the streaming kernel)
    uint32_t spin_limit;        // poll budget of those waits
    int n_base, ncols;          // streaming kernel: the columns [n_base, n_base + ncols) of this launch
};

// One element of row k of W (the A4 operand) at column n: from the fp16 copy,
// a kept row, or the dequantized codes.
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

}  // namespace llmint8
