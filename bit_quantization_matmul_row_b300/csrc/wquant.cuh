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

// Prefill operand of A3: int8 codes as exact fp16 integers in a per-call
// scratch of the same layout, which the tensor-core GEMM loads by TMA (sm_103a
// has no int8 tcgen05 MMA; kind::f16 on exact integer codes stands in).  Used
// for the weight codes Wq [N, K] and, by llmint8_gemm_i32, for caller codes of X.
//
// A bandwidth pass that keeps the load/store path of the SMs out of the way:
// bulk copies (TMA engine) bring 16 KB slices of the codes into shared memory,
// they are widened there into an output buffer, and a bulk store writes that
// back.  One CTA per SM, grid-strided over slices; the CTA runs two independent
// groups of four warps, each with its own ring of kWidenIn input and kWidenOut
// output buffers and its own named barrier, taking the CTA's slices in turn, so
// that one group widens while the other waits for data, fences or stores.  The
// codes may be read before the predecessor finishes only when they are
// constant (weights); the scratch is written only after it (the previous
// call's GEMM may still read it).  Waits are bounded: a timeout records the
// error word and the group stops after letting its copies in flight finish.
constexpr uint32_t kWidenChunk = 16384;  // int8 bytes per slice
constexpr int kWidenGroups = 2, kWidenIn = 3, kWidenOut = 2, kWidenThreads = 256;
constexpr int kWidenGroupThreads = kWidenThreads / kWidenGroups;
constexpr size_t kWidenGroupBytes = (size_t)kWidenIn * kWidenChunk + (size_t)kWidenOut * 2 * kWidenChunk;
constexpr size_t kWidenSmem = 1024 + kWidenGroups * kWidenGroupBytes + 256;
static_assert(kWidenSmem <= 232448, "one CTA per SM within the opt-in shared memory limit");

__global__ void __launch_bounds__(kWidenThreads, 1)
    k_widen_codes(const int8_t* __restrict__ src, __half* __restrict__ dst, size_t nbytes, int src_constant,
                  WsHeader* err, uint32_t spin_limit) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x;
    const int grp = tid / kWidenGroupThreads, gtid = tid % kWidenGroupThreads;
    uint8_t* in = sm + (size_t)grp * kWidenGroupBytes;                // [kWidenIn][kWidenChunk]
    uint8_t* out = in + (size_t)kWidenIn * kWidenChunk;               // [kWidenOut][2 * kWidenChunk]
    uint64_t* full_all = reinterpret_cast<uint64_t*>(sm + kWidenGroups * kWidenGroupBytes);
    uint64_t* full = full_all + grp * kWidenIn;                       // this group's [kWidenIn]
    __shared__ uint32_t s_ok[kWidenGroups];
    const size_t nchunks = (nbytes + kWidenChunk - 1) / kWidenChunk;
    // the group's slices: the CTA's slices blockIdx.x + i * gridDim.x with i = grp, grp + 2, ...
    auto chunk_of = [&](size_t j) { return (size_t)blockIdx.x + (j * kWidenGroups + grp) * gridDim.x; };
    auto bytes_of = [&](size_t c) {
        const size_t rest = nbytes - c * kWidenChunk;
        return (uint32_t)(rest < kWidenChunk ? rest : kWidenChunk);
    };
    auto issue = [&](size_t j) {  // group leader: slice j of the group into ring slot j % kWidenIn
        const size_t c = chunk_of(j);
        if (c >= nchunks) return;
        uint64_t* bar = &full[j % kWidenIn];
        mbar_arrive_expect_tx(bar, bytes_of(c));
        bulk_load_1d(in + (j % kWidenIn) * kWidenChunk, src + c * kWidenChunk, bytes_of(c), bar);
    };
    auto group_sync = [&]() { asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "n"(kWidenGroupThreads) : "memory"); };
    if (tid == 0) {
        for (int i = 0; i < kWidenGroups * kWidenIn; ++i) mbar_init(&full_all[i], 1);
        fence_mbar_init();
        for (int g = 0; g < kWidenGroups; ++g) s_ok[g] = 1u;
    }
    __syncthreads();
    pdl_trigger();
    if (!src_constant) pdl_wait();
    if (gtid == 0)
        for (int i = 0; i < kWidenIn; ++i) issue(i);
    pdl_wait();
    size_t j = 0;
    for (; chunk_of(j) < nchunks; ++j) {
        const size_t c = chunk_of(j);
        const int si = (int)(j % kWidenIn), so = (int)(j % kWidenOut);
        if (gtid == 0) {
            // the output slot's previous bulk store has finished reading it
            if (j >= (size_t)kWidenOut) bulk_wait_read<kWidenOut - 1>();
            s_ok[grp] = mbar_wait_bounded(&full[si], (uint32_t)(j / kWidenIn) & 1u, spin_limit, nullptr) ? 1u : 0u;
        }
        group_sync();
        if (!s_ok[grp]) break;
        const uint32_t nb = bytes_of(c);
        const uint8_t* a = in + (size_t)si * kWidenChunk;
        uint8_t* o = out + (size_t)so * 2 * kWidenChunk;
#pragma unroll 4
        for (uint32_t p = gtid * 16; p < nb; p += kWidenGroupThreads * 16) {
            const uint4 v = *reinterpret_cast<const uint4*>(a + p);
            uint32_t h[8];
            s8x4_to_half2x2(v.x, h[0], h[1]);
            s8x4_to_half2x2(v.y, h[2], h[3]);
            s8x4_to_half2x2(v.z, h[4], h[5]);
            s8x4_to_half2x2(v.w, h[6], h[7]);
            *reinterpret_cast<uint4*>(o + 2 * p) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(o + 2 * p + 16) = make_uint4(h[4], h[5], h[6], h[7]);
        }
        fence_proxy_async_smem();  // the bulk store reads these writes through the async proxy
        group_sync();
        if (gtid == 0) {
            bulk_store_1d(dst + c * kWidenChunk, o, 2 * nb);
            bulk_commit();
            issue(j + kWidenIn);  // the input slot is free again (the group passed the barrier)
        }
    }
    if (gtid == 0) {
        if (!s_ok[grp]) {
            record_error(err, kStatusTimeout, 30);
            // let the loads already issued land before shared memory goes away
            for (size_t k = j; k < j + kWidenIn && chunk_of(k) < nchunks; ++k)
                mbar_wait_bounded(&full[k % kWidenIn], (uint32_t)(k / kWidenIn) & 1u, 1u << 20, nullptr);
        }
        bulk_wait_all();
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
