// Prefill path (M > 16) of the LLM.int8() matmul: steps A3-A5 on the 5th-
// generation tensor cores.
//
// sm_103a has no int8 tcgen05 MMA (kind::i8 exists only on sm_100a/sm_110a),
// and its int8 mma.sync rate is ~140 TOPS.  The int8 codes are therefore fed to
// tcgen05.mma kind::f16 as exact fp16 integers.  Each product is an integer of
// magnitude <= 127^2 = 16129 and each partial sum over at most 1024 products
// stays below 2^24, so the fp32 TMEM accumulator holds it exactly.  The K loop
// is cut into chunks of at most 1024 (16 steps of 64) and equal length; each
// chunk is accumulated into one of two TMEM buffers and the epilogue warps
// drain it into int32 registers while the tensor core fills the other buffer.
// The integer product C is thus exact for any K (A3).
//
// The fp16 outlier slice (A4: X[:, O] . W16[O, :], fp32 accumulate) is one more
// chunk of the same pipeline, fed from the gathered operands Xo [M, Kp] and
// W16oT [N, Kp]; it stays in fp32.  The epilogue then computes
// Y = fp16(C * s_x[i] * s_w[n] / 127^2 + F) (A5) into registers, frees the
// TMEM buffer at once (the tensor core is already on the next tile and needs
// it one chunk later), and writes Y through a shared-memory staging buffer
// with TMA tensor stores: whole 128-byte row segments instead of one 16-byte
// piece per thread and row, which had flooded the L2 with partial-sector
// writes and slowed the operand loads of the next tile.
//
// Roles (320 threads, one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0      TMA producer: 4-stage ring of (A 128x64, B 256x64) fp16 tiles
//   warp 1      TMEM owner and MMA issuer (one thread), M=128 N=256 K=16 MMAs
//   warps 2..9  epilogue: warp w reads TMEM lanes 32*(w%4).., column half (w-2)/4,
//               and stores its 32 rows through its own 4 KB staging buffer
//
// PAIR (M > 128): the CTAs run as clusters of two that compute 256 x 256 tiles
// with tcgen05.mma.cta_group::2.  Each CTA loads its own 128 rows of A and its
// 128 columns of B, so a ring stage is 32 KB instead of 48 KB and the same
// shared memory holds 6 stages instead of 4.  The tensor core consumes a stage
// in about 0.3 us; with 4 stages its issuer waited for data about a third of
// the time (L2 latency under load), 6 stages cover 1.5 times as much.  Both
// producers' copies complete on the first CTA's full barrier (TMA
// .cta_group::2; that CTA registers the bytes of both), its MMA
// thread issues the M=256 N=256 MMAs, and its commits arrive on the empty and
// TMEM-full barriers of both CTAs (multicast).  Each CTA's epilogue drains its
// own TMEM (rows 0..127 of the pair tile in the first CTA, 128..255 in the
// second) and releases a TMEM buffer on the first CTA's barrier.
#pragma once

#include "common.cuh"
#include "xpass.cuh"

namespace llmint8 {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;      // one CTA per tile: 48 KB stages
constexpr int kPairStages = 6;  // CTA pairs: 32 KB stages
constexpr int kMaxStages = 8;   // CTA pairs on 256 x 128 tiles: 24 KB stages
constexpr int kChunkSteps = 16;  // 16 x 64 = 1024 products per exact fp32 chunk
constexpr int kEpiWarps = 8;
constexpr int kGemmThreads = 64 + kEpiWarps * 32;
constexpr uint32_t kStageA = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kStageB = kBN * kBK * 2;  // 32 KB
constexpr uint32_t kPairStageB = kStageB / 2;  // 16 KB: the CTA's half of the B tile
constexpr uint32_t kTmemCols = 512;          // two 256-column fp32 accumulators
static_assert(kStages * (kStageA + kStageB) == kPairStages * (kStageA + kPairStageB), "same ring size");
// After the ring: the barriers (1 KB block), then one output staging buffer per
// epilogue warp: 32 rows x 128 bytes, the box of a TMA store with the 128-byte
// swizzle (64 fp16 or 32 int32 columns of the warp's 32 rows).
constexpr uint32_t kOutStage = 32 * 128;
constexpr size_t kGemmSmem =
    1024 /*align slack*/ + (size_t)kStages * (kStageA + kStageB) + 1024 + (size_t)kEpiWarps * kOutStage;
static_assert(kGemmSmem <= 232448, "shared memory of one CTA");

// Ring depth and B bytes per stage of one CTA for a tile width BN (256, or 128
// when wide tiles would leave SMs idle): the rings fill the same 192 KB.
__host__ __device__ constexpr int gemm_stages(bool pair, int BN) {
    return !pair ? (BN == 256 ? kStages : kPairStages) : BN == 256 ? kPairStages : 8;
}
__host__ __device__ constexpr uint32_t gemm_stage_b(bool pair, int BN) {
    return (uint32_t)(pair ? BN / 2 : BN) * kBK * 2;
}
static_assert(gemm_stages(true, 128) * (kStageA + gemm_stage_b(true, 128)) == kStages * (kStageA + kStageB) &&
                  gemm_stages(false, 128) * (kStageA + gemm_stage_b(false, 128)) == kStages * (kStageA + kStageB),
              "same ring size");

struct GemmArgs {
    const float* row_scale;  // [M]
    const float* col_scale;  // [N]
    const WsHeader* hdr;     // outlier_count
    WsHeader* err;           // error word
    int M, N, K;
    int use_outliers;
    uint32_t spin_limit;
};

struct GemmSmem {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t teardown;
    uint32_t tmem_base;
    uint32_t abort_flag;
};

template <bool WRITE_I32, bool PAIR, typename T, int BN = kBN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
              const __grid_constant__ CUtensorMap tm_xo, const __grid_constant__ CUtensorMap tm_wo,
              const __grid_constant__ CUtensorMap tm_out, GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    static_assert(BN == kBN || BN == 128, "tile widths: 256 or 128");
    constexpr int S = gemm_stages(PAIR, BN);
    constexpr uint32_t SB = gemm_stage_b(PAIR, BN);  // B bytes of a stage in this CTA
    constexpr uint32_t TC = 2 * BN;                  // TMEM columns: two fp32 accumulators
    constexpr int HC = BN / 2;                       // columns drained by one epilogue warp
    uint8_t* stage_a = smem;
    uint8_t* stage_b = smem + S * kStageA;
    GemmSmem* ss = reinterpret_cast<GemmSmem*>(smem + S * (kStageA + SB));
    static_assert(sizeof(GemmSmem) <= 1024, "barrier block");
    uint8_t* stage_out = smem + S * (kStageA + SB) + 1024;  // 1024-aligned, as the swizzle needs
    volatile uint32_t* abort_flag = &ss->abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // work units: 128 x 256 tiles, or 256 x 256 tiles of a CTA pair
    const uint32_t rank = PAIR ? cluster_cta_rank() : 0u;
    const int unit_rows = PAIR ? 2 * kBM : kBM;
    const int tiles_m = (a.M + unit_rows - 1) / unit_rows, tiles_n = (a.N + BN - 1) / BN;
    const int ntiles = tiles_m * tiles_n;
    const int unit0 = PAIR ? (int)blockIdx.x / 2 : (int)blockIdx.x;
    const int ustride = PAIR ? (int)gridDim.x / 2 : (int)gridDim.x;
    // this CTA's first row in unit row tm and first column of its B half
    auto row_of = [&](int tm) { return tm * unit_rows + (int)rank * kBM; };
    auto bcol_of = [&](int tn) { return tn * BN + (int)rank * (BN / 2); };
    const int ksteps = (a.K + kBK - 1) / kBK;
    const int nchunks_int = (ksteps + kChunkSteps - 1) / kChunkSteps;

    // set-up that does not depend on the X pass overlaps its tail (programmatic
    // dependent launch); everything after pdl_wait() may read its results
    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&ss->full[s], 1);
            mbar_init(&ss->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ss->tmem_full[b], 1);
            mbar_init(&ss->tmem_empty[b], PAIR ? 2 * kEpiWarps : kEpiWarps);
        }
        mbar_init(&ss->teardown, 1);
        ss->abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
        tma_prefetch_desc(&tm_out);
        if (a.use_outliers) {
            tma_prefetch_desc(&tm_xo);
            tma_prefetch_desc(&tm_wo);
        }
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(&ss->tmem_base, TC);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&ss->tmem_base, TC);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync_all();  // both CTAs' barriers initialised before any remote arrive
    tc_fence_after();
    // barriers of the pair's first CTA, as shared::cluster addresses
    const uint32_t lead_full0 = PAIR ? mapa_shared(smem_u32(&ss->full[0]), 0) : 0u;
    const uint32_t lead_tmem_empty0 = PAIR ? mapa_shared(smem_u32(&ss->tmem_empty[0]), 0) : 0u;
    const uint32_t tmem_base = ss->tmem_base;
    pdl_wait();
    const int n_out = a.use_outliers ? __ldcg(&a.hdr->outlier_count) : 0;
    const int osteps = (n_out + kBK - 1) / kBK;

    auto wait_bar = [&](uint64_t* bar, uint32_t parity) -> bool {
        return mbar_wait_bounded(bar, parity, a.spin_limit, abort_flag);
    };
    auto fail = [&](uint32_t where) {
        *abort_flag = 1u;
        record_error(a.err, kStatusTimeout, where);
    };
    // whole-warp bounded wait: lane 0 polls, the result is broadcast, and the
    // warp is converged again for the .sync.aligned TMEM loads that follow
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        uint32_t got = 0;
        if (lane == 0) got = wait_bar(bar, parity) ? 1u : 0u;
        got = __shfl_sync(0xffffffffu, got, 0);
        return got != 0;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_parity[S];
            bool issued[S];
            for (int s = 0; s < S; ++s) issued[s] = false, issued_parity[s] = 0;
            bool ok = true;
            for (int tile = unit0; tile < ntiles && ok; tile += ustride) {
                const int tm = tile % tiles_m, tn = tile / tiles_m;
                const int total = ksteps + osteps;
                for (int s = 0; s < total; ++s) {
                    if (!wait_bar(&ss->empty[stage], phase ^ 1u)) {
                        fail(1);
                        ok = false;
                        break;
                    }
                    const bool main_k = s < ksteps;
                    const int kx = (main_k ? s : s - ksteps) * kBK;
                    const void* ta = main_k ? (const void*)&tm_a : (const void*)&tm_xo;
                    const void* tb = main_k ? (const void*)&tm_b : (const void*)&tm_wo;
                    if constexpr (PAIR) {
                        // this CTA's rows of A and columns of B, signalled on the first CTA's
                        // barrier, where the first CTA alone registers both CTAs' bytes (the
                        // other CTA's copies may land first: the transaction count of the
                        // phase goes negative until the arrival, which completes nothing)
                        const uint32_t fb = lead_full0 + (uint32_t)stage * 8u;
                        if (rank == 0) mbar_arrive_expect_tx(&ss->full[stage], 2 * (kStageA + SB));
                        tma_load_2d_pair(stage_a + stage * kStageA, ta, fb, kx, row_of(tm));
                        tma_load_2d_pair(stage_b + stage * SB, tb, fb, kx, bcol_of(tn));
                    } else {
                        mbar_arrive_expect_tx(&ss->full[stage], kStageA + SB);
                        tma_load_2d(stage_a + stage * kStageA, ta, &ss->full[stage], kx, tm * kBM);
                        tma_load_2d(stage_b + stage * SB, tb, &ss->full[stage], kx, tn * BN);
                    }
                    issued[stage] = true;
                    issued_parity[stage] = phase;
                    if (++stage == S) stage = 0, phase ^= 1u;
                }
            }
            if (!ok && !PAIR) {
                // let copies already in flight land before the CTA can exit
                // (pairs: they signal the first CTA, which keeps running until
                // the cluster barrier at the end)
                for (int s = 0; s < S; ++s)
                    if (issued[s]) mbar_wait_bounded(&ss->full[s], issued_parity[s], 1u << 20, nullptr);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // (pairs: the first CTA's thread issues for both)
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = make_idesc_f16(PAIR ? 2 * kBM : kBM, BN);
            // the outlier chunk multiplies the gathered X and W values, of format T
            constexpr uint32_t idesc_o = make_idesc_f16(PAIR ? 2 * kBM : kBM, BN, Fmt<T>::kBF16);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t chunk = 0;
            bool ok = true;
            for (int tile = unit0; tile < ntiles && ok; tile += ustride) {
                const int nchunks = nchunks_int + (osteps ? 1 : 0);
                for (int ch = 0; ch < nchunks && ok; ++ch, ++chunk) {
                    const uint32_t b = chunk & 1u, use = (chunk >> 1) & 1u;
                    if (!wait_bar(&ss->tmem_empty[b], use ^ 1u)) {
                        fail(2);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // the K steps in nchunks_int chunks of equal length (+-1, at most
                    // 16): no short tail chunk whose drain outlasts its MMAs
                    const bool int_chunk = ch < nchunks_int;
                    const int s_begin = int_chunk ? ch * ksteps / nchunks_int : ksteps;
                    const int s_end = int_chunk ? (ch + 1) * ksteps / nchunks_int : ksteps + osteps;
                    const uint32_t d_tmem = tmem_base + b * (uint32_t)BN;
                    const uint32_t id = int_chunk ? idesc : idesc_o;
                    for (int s = s_begin; s < s_end; ++s) {
                        if (!wait_bar(&ss->full[stage], phase)) {
                            fail(3);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t ad = make_sdesc_k128(smem_u32(stage_a + stage * kStageA));
                        const uint64_t bd = make_sdesc_k128(smem_u32(stage_b + stage * SB));
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            // advance 16 fp16 = 32 bytes inside the 128-byte swizzled row
                            const uint32_t acc = (s > s_begin || kk > 0) ? 1u : 0u;
                            if constexpr (PAIR)
                                tc_mma_f16_pair(d_tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), id, acc);
                            else
                                tc_mma_f16(d_tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), id, acc);
                        }
                        if constexpr (PAIR)
                            tc_commit_pair(&ss->empty[stage], 0x3);  // both CTAs' stage is free
                        else
                            tc_commit(&ss->empty[stage]);
                        if (++stage == S) stage = 0, phase ^= 1u;
                    }
                    if (ok) {
                        if constexpr (PAIR)
                            tc_commit_pair(&ss->tmem_full[b], 0x3);
                        else
                            tc_commit(&ss->tmem_full[b]);
                    }
                }
            }
            // all issued MMAs complete before TMEM can be released
            if constexpr (PAIR)
                tc_commit_pair(&ss->teardown, 0x1);
            else
                tc_commit(&ss->teardown);
            mbar_wait_bounded(&ss->teardown, 0, a.spin_limit, nullptr);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 2;
        const int q = warp & 3;          // TMEM lane quarter this warp may access
        const int h = ew >> 2;           // column half of the 256-wide tile
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        uint32_t chunk = 0;
        bool ok = true;
        // release a TMEM buffer: on this CTA's barrier, or the first CTA's for pairs
        auto release = [&](uint32_t b) {
            if constexpr (PAIR)
                mbar_arrive_cluster(lead_tmem_empty0 + b * 8u);
            else
                mbar_arrive(&ss->tmem_empty[b]);
        };
        // This warp's output staging buffer.  At the start of a tile its first
        // HC floats receive the column scales of the warp's columns; once the
        // values of the tile are in registers it receives one TMA box of output
        // at a time: row r (= lane) as eight 16-byte chunks, chunk k at position
        // k ^ (r % 8) (the 128-byte swizzle).
        uint8_t* stg = stage_out + ew * kOutStage;
        const float* cs = reinterpret_cast<const float*>(stg);
        auto stage_row = [&](int k, uint4 v) {
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((k ^ (lane & 7)) << 4)) = v;
        };
        // publish the staged box to the async proxy and store it; the next
        // writer of the buffer waits for the store to have read it
        auto store_box = [&](int x, int y0) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && x < a.N && y0 < a.M) {
                tma_store_2d(&tm_out, stg, x, y0);
                bulk_commit();
            }
        };
        auto buffer_free = [&]() {
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
        };
        for (int tile = unit0; tile < ntiles && ok; tile += ustride) {
            const int tm = tile % tiles_m, tn = tile / tiles_m;
            const int row0 = row_of(tm) + q * 32;  // first of this warp's 32 rows
            const int row = row0 + lane;
            const int col0 = tn * BN + h * HC;
            buffer_free();
            if constexpr (!WRITE_I32) {
                // read once per tile, while the tensor core works on the first
                // chunk (N is a multiple of 16: whole float4s)
                float* csw = reinterpret_cast<float*>(stg);
                for (int c = lane * 4; c < HC; c += 128) {
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (col0 + c < a.N) v = __ldg(reinterpret_cast<const float4*>(a.col_scale + col0 + c));
                    *reinterpret_cast<float4*>(csw + c) = v;
                }
                __syncwarp();
            }
            // Exact conversion of a chunk's integer-valued fp32 sums v: for |v| <=
            // 2^22, v + 1.5 * 2^23 is a float of exponent 23 whose bit pattern is
            // 0x4B400000 + v.  The int32 sum adds these patterns and starts from
            // -nchunks * 0x4B400000 (mod 2^32), which leaves the exact integer.  A
            // batch of 16 in which some |v| reaches 2^22 (possible only close to the
            // 2^24 bound of a chunk) is converted by cvt.rni instead, for the whole warp.
            uint32_t sum[HC];
            const uint32_t bias = 0u - (uint32_t)nchunks_int * 0x4B400000u;
#pragma unroll
            for (int c = 0; c < HC; ++c) sum[c] = bias;
            for (int ch = 0; ch < nchunks_int; ++ch, ++chunk) {
                const uint32_t b = chunk & 1u, use = (chunk >> 1) & 1u;
                const bool got = warp_wait(&ss->tmem_full[b], use);
                if (!got) {
                    if (lane == 0) fail(4);
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < HC / 16; ++j) {
                    uint32_t r[16];
                    tmem_ld_32x32b_x16(tmem_base + lane_base + b * BN + h * HC + j * 16, r);
                    tmem_ld_wait();
                    float mx = 0.f;
#pragma unroll
                    for (int c = 0; c < 16; ++c) mx = fmaxf(mx, fabsf(__uint_as_float(r[c])));
                    if (__any_sync(0xffffffffu, mx >= 4194304.0f)) {
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            sum[j * 16 + c] += (uint32_t)__float2int_rn(__uint_as_float(r[c])) + 0x4B400000u;
                    } else {
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            sum[j * 16 + c] += __float_as_uint(__fadd_rn(__uint_as_float(r[c]), 12582912.0f));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release(b);
            }
            if (!ok) break;
            uint32_t fb = 0;
            const bool has_f = osteps > 0;
            if (has_f) {
                fb = chunk & 1u;
                const uint32_t use = (chunk >> 1) & 1u;
                if (!warp_wait(&ss->tmem_full[fb], use)) {
                    if (lane == 0) fail(5);
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            // the fp32 accumulator is released as soon as its values are in
            // registers; the stores of the tile follow
            auto release_final = [&]() {
                if (has_f) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) release(fb);
                    ++chunk;
                }
            };
            if constexpr (WRITE_I32) {
                release_final();  // C alone: the outlier chunk is not run for int32 output
#pragma unroll
                for (int p = 0; p < HC / 32; ++p) {  // boxes of 32 int32 columns
                    if (p > 0) buffer_free();
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        stage_row(k, make_uint4(sum[p * 32 + k * 4], sum[p * 32 + k * 4 + 1], sum[p * 32 + k * 4 + 2],
                                                sum[p * 32 + k * 4 + 3]));
                    store_box(col0 + p * 32, row0);
                }
            } else {
                const float sx = row < a.M ? __ldcg(a.row_scale + row) * (1.0f / 16129.0f) : 0.0f;
                uint32_t o[HC / 2];  // Y values, two per word
#pragma unroll
                for (int j = 0; j < HC / 16; ++j) {
                    uint32_t r[16];
                    if (has_f) {
                        tmem_ld_32x32b_x16(tmem_base + lane_base + fb * BN + h * HC + j * 16, r);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int c = 0; c < 16; ++c) r[c] = 0u;
                    }
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const float4 s4 = *reinterpret_cast<const float4*>(cs + j * 16 + v * 4);
                        const int c = j * 16 + v * 4;
                        const float y0 = fmaf((float)(int32_t)sum[c], sx * s4.x, __uint_as_float(r[v * 4]));
                        const float y1 = fmaf((float)(int32_t)sum[c + 1], sx * s4.y, __uint_as_float(r[v * 4 + 1]));
                        const float y2 = fmaf((float)(int32_t)sum[c + 2], sx * s4.z, __uint_as_float(r[v * 4 + 2]));
                        const float y3 = fmaf((float)(int32_t)sum[c + 3], sx * s4.w, __uint_as_float(r[v * 4 + 3]));
                        o[c / 2] = Fmt<T>::pack2(y0, y1);
                        o[c / 2 + 1] = Fmt<T>::pack2(y2, y3);
                    }
                }
                release_final();
                __syncwarp();  // every lane has read the column scales
#pragma unroll
                for (int p = 0; p < HC / 64; ++p) {  // boxes of 64 fp16 columns
                    if (p > 0) buffer_free();
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        stage_row(k, make_uint4(o[p * 32 + k * 4], o[p * 32 + k * 4 + 1], o[p * 32 + k * 4 + 2],
                                                o[p * 32 + k * 4 + 3]));
                    store_box(col0 + p * 64, row0);
                }
            }
        }
        // stores in flight complete before the CTA exits
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    // pairs: the first CTA's MMAs into both TMEMs have completed (its issuer
    // waited for the teardown commit) before either CTA frees its columns
    if constexpr (PAIR) cluster_sync_all();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, TC);
        else
            tmem_dealloc(tmem_base, TC);
    }
}

}  // namespace llmint8
