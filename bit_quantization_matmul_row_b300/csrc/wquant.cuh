// A0: weight quantization, once per weight matrix (paper walkthrough, section
// 2.1: one scale per output column of W; Lightning Fabric 8-bit page, section
// 2.2: per output channel).  The column absmax covers all K rows.
//
//   colScaleW[n] = max_k |W[k,n]|
//   Wq[n, k]     = round-half-away(fp32(W[k,n] * fp32(127 / colScaleW[n])))
//
// W is [K, N] row-major; Wq is transposed to [N, K] (K contiguous): the layout
// both product paths stream.  Wq is the only code copy kept: the prefill path
// widens it into a per-call fp16 scratch (k_widen_codes) for the tensor cores.
#pragma once

#include "common.cuh"

namespace llmint8 {

// Column absmax, pass 1: each CTA reduces a 256-column strip over a slice of
// rows and folds its result into colScaleW with an integer atomicMax (valid for
// non-negative floats).  colScaleW must be zero on entry.
template <typename T>
__global__ void __launch_bounds__(256) k_col_absmax(const __half* __restrict__ W, int K, int N,
                                                    float* __restrict__ col_amax) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c0 = blockIdx.x * 256 + lane * 8;
    float m[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (c0 < N) {
        for (int r = blockIdx.y * 8 + warp; r < K; r += gridDim.y * 8) {
            const uint4 v = ldg_nc_v4(W + (size_t)r * N + c0);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = Fmt<T>::to_float2(w[e]);
                m[2 * e] = fmaxf(m[2 * e], fabsf(f.x));
                m[2 * e + 1] = fmaxf(m[2 * e + 1], fabsf(f.y));
            }
        }
    }
    __shared__ float s[8][256];
#pragma unroll
    for (int e = 0; e < 8; ++e) s[warp][lane * 8 + e] = m[e];
    __syncthreads();
    const int c = blockIdx.x * 256 + threadIdx.x;
    float r = s[0][threadIdx.x];
#pragma unroll
    for (int w = 1; w < 8; ++w) r = fmaxf(r, s[w][threadIdx.x]);
    if (c < N && r > 0.0f) atomicMax(reinterpret_cast<int*>(col_amax) + c, __float_as_int(r));
}

// Pass 2: quantize a 64(k) x 64(n) tile and write it transposed.
template <typename T>
__global__ void __launch_bounds__(256) k_quantize_weight_tile(const __half* __restrict__ W, int K, int N,
                                                              const float* __restrict__ col_amax,
                                                              int8_t* __restrict__ Wq) {
    __shared__ float s_sf[64];
    __shared__ int8_t tile[64][64 + 4];  // [n][k]
    const int k0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    const int tid = threadIdx.x;
    if (tid < 64) {
        const int n = n0 + tid;
        const float amax = n < N ? col_amax[n] : 0.0f;
        s_sf[tid] = amax > 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
    }
    __syncthreads();
    // read: 64 rows (k) x 64 columns (n), 2 columns per thread-iteration
    for (int e = tid; e < 64 * 32; e += 256) {
        const int kr = e >> 5, nc = (e & 31) * 2;
        const int k = k0 + kr, n = n0 + nc;
        if (k < K && n < N) {  // N % 16 == 0: n and n+1 both valid
            const float2 f = Fmt<T>::to_float2(*reinterpret_cast<const uint32_t*>(W + (size_t)k * N + n));
            const float q0 = fminf(fmaxf(roundf(__fmul_rn(f.x, s_sf[nc])), -127.0f), 127.0f);
            const float q1 = fminf(fmaxf(roundf(__fmul_rn(f.y, s_sf[nc + 1])), -127.0f), 127.0f);
            tile[nc][kr] = (int8_t)(int)q0;
            tile[nc + 1][kr] = (int8_t)(int)q1;
        }
    }
    __syncthreads();
    // write: row n, 64 consecutive k; 4 codes per thread-iteration
    for (int e = tid; e < 64 * 16; e += 256) {
        const int nr = e >> 4, kc = (e & 15) * 4;
        const int n = n0 + nr, k = k0 + kc;
        if (n < N && k < K) {  // K % 16 == 0: all 4 valid
            const int8_t c0 = tile[nr][kc], c1 = tile[nr][kc + 1], c2 = tile[nr][kc + 2], c3 = tile[nr][kc + 3];
            const uint32_t packed = (uint32_t)(uint8_t)c0 | ((uint32_t)(uint8_t)c1 << 8) |
                                    ((uint32_t)(uint8_t)c2 << 16) | ((uint32_t)(uint8_t)c3 << 24);
            *reinterpret_cast<uint32_t*>(Wq + (size_t)n * K + k) = packed;
        }
    }
}

// Prefill operand of A3: the int8 codes Wq [N, K] as exact fp16 integers in a
// per-call scratch of the same layout, which the tensor-core GEMM loads by TMA
// (sm_103a has no int8 tcgen05 MMA; kind::f16 on exact integer codes stands in).
// Each thread widens kWidenUnroll 16-code chunks per step (all loads issued
// before the stores, grid-strided so that a warp touches 512 contiguous bytes).
// The scratch is in the workspace, which the previous call's GEMM may still be
// reading: the stores wait for the predecessor (programmatic dependent launch).
constexpr int kWidenUnroll = 4;
__global__ void __launch_bounds__(256, 8) k_widen_codes(const int8_t* __restrict__ Wq, __half* __restrict__ out,
                                                     size_t n16) {
    pdl_trigger();
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    bool waited = false;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += kWidenUnroll * stride) {
        uint4 v[kWidenUnroll];
#pragma unroll
        for (int u = 0; u < kWidenUnroll; ++u) {
            const size_t c = i + u * stride;
            v[u] = c < n16 ? ldg_nc_v4(Wq + c * 16) : make_uint4(0u, 0u, 0u, 0u);
        }
        if (!waited) {
            pdl_wait();
            waited = true;
        }
#pragma unroll
        for (int u = 0; u < kWidenUnroll; ++u) {
            const size_t c = i + u * stride;
            if (c < n16) {
                uint32_t h[8];
                s8x4_to_half2x2(v[u].x, h[0], h[1]);
                s8x4_to_half2x2(v[u].y, h[2], h[3]);
                s8x4_to_half2x2(v[u].z, h[4], h[5]);
                s8x4_to_half2x2(v[u].w, h[6], h[7]);
                uint4* o = reinterpret_cast<uint4*>(out + c * 16);
                o[0] = make_uint4(h[0], h[1], h[2], h[3]);
                o[1] = make_uint4(h[4], h[5], h[6], h[7]);
            }
        }
    }
}

// Kept fp16 rows of W (A4 without a full fp16 copy): row_map[k] = -1 for all k,
// then for each listed row r: W16c[r, :] = W16[rows[r], :] and row_map[rows[r]] = r.
// A listed row outside [0, K) gets a zero row and no map entry.
__global__ void __launch_bounds__(256) k_row_map_clear(int32_t* __restrict__ row_map, int K) {
    for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < K; k += gridDim.x * blockDim.x) row_map[k] = -1;
}

__global__ void __launch_bounds__(256) k_pack_w16_rows(const __half* __restrict__ W16, int K, int N,
                                                       const int32_t* __restrict__ rows, int nrows,
                                                       __half* __restrict__ W16c, int32_t* __restrict__ row_map) {
    const int vec = N / 8;  // 16-byte vectors per row
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < (size_t)nrows * vec;
         e += (size_t)gridDim.x * blockDim.x) {
        const int r = (int)(e / vec), v = (int)(e - (size_t)r * vec);
        const int k = rows[r];
        const bool ok = k >= 0 && k < K;
        const uint4 val = ok ? ldg_nc_v4(W16 + (size_t)k * N + 8 * v) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(W16c + (size_t)r * N + 8 * v) = val;
        if (ok && v == 0) row_map[k] = r;
    }
}

}  // namespace llmint8
