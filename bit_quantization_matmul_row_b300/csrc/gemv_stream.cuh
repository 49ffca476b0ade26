// Decode path (M <= 16) of the LLM.int8() matmul: steps A3-A5 in one persistent
// streaming kernel.
//
// Decode is bound by streaming the int8 weight codes from HBM once (every
// decode step reads all weights: INT8-vs-FP8 page, section 1).  On B300 a
// 17-45 MB stream reaches the HBM rate only when every SM keeps well over
// 100 KB in flight from its first microsecond, in few large copies, and when
// one call's stream starts before the previous call's kernels have drained.
// Hence:
//
//  * one CTA per SM (grid = min(tiles, SMs)); CTA b owns a contiguous run of
//    16-column tiles, hence a contiguous column range of Y;
//  * one producer thread moves each int8 stage with ONE tensor load per
//    operand: Wq [N, K] is viewed as a 3D tensor (64 bytes of K, rows with
//    stride K, 64-byte K steps with stride 64), so a box of (64, 16, SK/64)
//    lands as [SK/64 steps][16 rows][64 bytes]; the X codes likewise as
//    [SK/64][M][64].  In that layout the 32 lanes' 16-byte reads fall on
//    distinct bank groups.  A ragged K (K % 64 != 0) has its last partial step
//    copied row by row into a small tail area of the stage;
//  * the weight halves of the first ring round are requested before
//    griddepcontrol.wait: they do not depend on the X pass, so under
//    programmatic dependent launch they stream while the X pass of the same
//    call still runs.  The X halves follow right after the wait on the same
//    barriers (mbarrier.expect_tx for the weights, arrive.expect_tx for X);
//  * 8 consumer warps share each stage's K steps.  Up to 2 rows of X use
//    dp4a (four int8 products per instruction, no padding rows); more rows use
//    the int8 mma.sync m16n8k32 (s8 x s8 -> s32), whose 8-row tiles pad M.
//    Both are exact integer arithmetic (A3);
//  * a tile ends with one barrier of the 8 warps (an mbarrier, bounded): their
//    partial sums become the tile's int32 C in shared memory while the producer
//    keeps the ring streaming;
//  * the fp16 outlier slice (A4) comes last, through the same ring: for a chunk
//    of outlier columns o the producer warp copies W16[o, columns of this CTA]
//    (one contiguous segment per o) and the gathered X values; the consumers
//    accumulate F for the CTA's whole column range (fp32);
//  * the final pass applies the scale outer product and adds F (A5), and
//    writes Y (or C).
//
// Every wait is bounded; on a timeout the error word is set, the other roles
// leave through the abort flag, and the producer waits for its copies in
// flight before the CTA ends.
#pragma once

#include "common.cuh"
#include "gemv.cuh"
#include "xpass.cuh"

namespace llmint8 {

constexpr int kGsWarps = 8;                      // consumer warps
constexpr int kGsThreads = (kGsWarps + 1) * 32;  // + one producer warp
constexpr int kGsCols = 16;                      // output columns of a tile
constexpr int kGsChunk = 64;                     // outlier columns per outlier stage (at most)
constexpr int kGsMaxStages = 8;
constexpr int kGsTilesMax = 16;                  // tiles per CTA and launch (wider N: several launches)
constexpr size_t kGsSmemBudget = 184 * 1024;     // ring + C/F buffers (dynamic shared memory)

// consumer arithmetic: dp4a for up to 2 rows of X, mma.sync with one or two
// 8-row tiles above
enum { kGsDp4a = 0, kGsMma1 = 1, kGsMma2 = 2 };
__host__ __device__ constexpr int gs_mode(int M) { return M <= 2 ? kGsDp4a : (M <= 8 ? kGsMma1 : kGsMma2); }
// K bytes of one stage: 2048 up to 8 rows of X, 1024 above (the X rows make a stage larger)
__host__ __device__ constexpr int gs_stage_k(int mode) { return mode == kGsMma2 ? 1024 : 2048; }

// Launch plan of one call (host-computed; shared-memory offsets in bytes)
struct GsPlan {
    int R;          // ring stages
    int SB;         // bytes of one stage
    int ns;         // int8 stages per tile
    int kfull;      // whole 64-byte K steps (K / 64)
    int tail;       // K % 64: bytes of the ragged last step (0: none)
    int tail_off;   // offset of the tail area inside a stage
    int tiles_max;  // most tiles one CTA owns
    int c_off;      // int32 C [tiles_max][M][16] after the ring
    int f_off;      // fp32 F [M][16 tiles_max] after C
};

__host__ __device__ inline GsPlan gs_plan(int M, int K, int N, int grid) {
    GsPlan p;
    const int mode = gs_mode(M), SK = gs_stage_k(mode);
    p.kfull = K / 64;
    p.tail = K % 64;
    const int steps = p.kfull + (p.tail ? 1 : 0);
    p.ns = (steps * 64 + SK - 1) / SK;
    p.tail_off = (kGsCols + M) * SK;
    p.SB = ((p.tail_off + (p.tail ? (kGsCols + M) * 64 : 0)) + 127) / 128 * 128;
    const int tiles = N / kGsCols;
    p.tiles_max = (tiles + grid - 1) / grid;
    const int cbytes = p.tiles_max * M * kGsCols * 4;
    int R = (int)((kGsSmemBudget - 2 * (size_t)cbytes) / p.SB);
    p.R = R > kGsMaxStages ? kGsMaxStages : R;
    p.c_off = p.R * p.SB;
    p.f_off = p.c_off + cbytes;
    return p;
}
__host__ __device__ inline size_t gs_smem_bytes(const GsPlan& p) { return 128 + (size_t)p.f_off + (p.f_off - p.c_off); }

struct GsBars {
    uint64_t full[kGsMaxStages];
    uint64_t empty[kGsMaxStages];
    uint64_t red[2];  // the 8 warps' partials of a tile are in s_red (tiles alternate)
    uint32_t abort_flag;
};

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* desc, uint64_t* bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(desc), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

template <int MODE, bool WRITE_I32, typename T>
__global__ void __launch_bounds__(kGsThreads, 1)
    k_gemv_stream(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx, GemvArgs a, GsPlan p) {
    constexpr int SK = gs_stage_k(MODE);
    constexpr int NST = SK / 64;                       // 64-byte K steps of a stage
    constexpr int MR = MODE == kGsMma2 ? 16 : 8;       // rows of the partial-sum buffer
    constexpr int NPART = MODE == kGsDp4a ? 4 : kGsWarps;  // partial sums per output
    __shared__ int32_t s_red[2][NPART][MR][kGsCols];
    __shared__ GsBars sb;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint8_t* ring = smem;
    int32_t* s_c = reinterpret_cast<int32_t*>(smem + p.c_off);  // [tiles][M][16]
    float* s_f = reinterpret_cast<float*>(smem + p.f_off);      // [M][cols]
    volatile uint32_t* abort_flag = &sb.abort_flag;

    const int M = a.M, K = a.K, N = a.N, R = p.R, SB = p.SB;
    const int ns = p.ns;
    // this launch covers columns [n_base, n_base + ncols) of Y
    const int tiles = a.ncols / kGsCols, G = gridDim.x, b = blockIdx.x;
    const int t_begin = (int)((long long)b * tiles / G);
    const int my_tiles = (int)((long long)(b + 1) * tiles / G) - t_begin;  // >= 1: G <= tiles
    const int cols = my_tiles * kGsCols, n_begin = a.n_base + t_begin * kGsCols;
    const int total = my_tiles * ns;  // int8 stages
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    pdl_trigger();
    if (tid == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(&sb.full[s], 1);
            mbar_init(&sb.empty[s], kGsWarps);
        }
        mbar_init(&sb.red[0], kGsWarps);
        mbar_init(&sb.red[1], kGsWarps);
        sb.abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tw);
        tma_prefetch_desc(&tx);
    }
    __syncthreads();
    auto fail = [&](uint32_t where) {
        record_error(a.hdr_err, kStatusTimeout, where);
        *abort_flag = 1u;
    };
    // outlier stages: chunk size such that a chunk's W16 segments and X values fit a stage
    const int seg = cols * 2;  // bytes of W16[o, this CTA's columns]
    int chunk = (SB - M * kGsChunk * 2) / seg;
    chunk = chunk > kGsChunk ? kGsChunk : (chunk & ~7);  // a multiple of 8: 16-byte X value copies

    if (warp == kGsWarps) {
        // ---------------------------------------------------------------- producer warp
        const bool leader = lane == 0;
        int j = 0, s = 0;  // tile and stage within it of the next int8 stage
        // bytes a stage receives: the whole tensor box (steps past K are filled
        // with zeros and count) when the stage starts inside K, plus the tail rows
        auto wbytes = [&](int st) {
            const bool has_tail = p.tail && st == p.kfull / NST;
            return (uint32_t)((st * NST < p.kfull ? kGsCols * SK : 0) + (has_tail ? kGsCols * p.tail : 0));
        };
        auto xbytes = [&](int st) {
            const bool has_tail = p.tail && st == p.kfull / NST;
            return (uint32_t)((st * NST < p.kfull ? M * SK : 0) + (has_tail ? M * p.tail : 0));
        };
        auto issue_w = [&](int q) {
            uint8_t* dst = ring + (size_t)q * SB;
            const int n0 = n_begin + j * kGsCols;
            if (s * NST < p.kfull) tma_load_3d(dst, &tw, &sb.full[q], 0, n0, s * NST);
            if (p.tail && s == p.kfull / NST) {
                const int8_t* src = a.Wq + (size_t)n0 * K + (size_t)p.kfull * 64;
                for (int r = 0; r < kGsCols; ++r)
                    bulk_load_1d(dst + p.tail_off + r * 64, src + (size_t)r * K, (uint32_t)p.tail, &sb.full[q]);
            }
        };
        auto issue_x = [&](int q, int st) {
            uint8_t* dst = ring + (size_t)q * SB;
            if (st * NST < p.kfull) tma_load_3d(dst + kGsCols * SK, &tx, &sb.full[q], 0, 0, st * NST);
            if (p.tail && st == p.kfull / NST) {
                const int8_t* src = a.codes + (size_t)p.kfull * 64;
                for (int i = 0; i < M; ++i)
                    bulk_load_1d(dst + p.tail_off + (kGsCols + i) * 64, src + (size_t)i * K, (uint32_t)p.tail,
                                 &sb.full[q]);
            }
        };
        // whole-warp bounded wait for the consumers' release of stage v's slot
        auto wait_slot = [&](int v) -> bool {
            uint32_t got = 1;
            if (v >= R) {
                if (leader)
                    got = mbar_wait_bounded(&sb.empty[v % R], (uint32_t)((v / R - 1) & 1), a.spin_limit, abort_flag)
                              ? 1u
                              : 0u;
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got && leader && !*abort_flag) fail(31);  // a wait that ran out, not consumers that left
            }
            return got != 0;
        };
        const int pre = min(R, total);
        int issued = 0;  // stages requested so far
        // first ring round: the weights only, before the dependency wait
        for (int u = 0; u < pre; ++u) {
            if (leader) {
                mbar_expect_tx(&sb.full[u], wbytes(s));
                issue_w(u);
            }
            if (++s == ns) s = 0, ++j;
        }
        issued = pre;
        pdl_wait();  // the X codes and the outlier list are written by the X pass
        if (leader)
            for (int u = 0; u < pre; ++u) {
                const int st = u % ns;
                mbar_arrive_expect_tx(&sb.full[u], xbytes(st));
                issue_x(u, st);
            }
        bool ok = true;
        for (int u = pre; u < total && ok; ++u) {
            if (!(ok = wait_slot(u))) break;
            if (leader) {
                const int q = u % R;
                mbar_arrive_expect_tx(&sb.full[q], wbytes(s) + xbytes(s));
                issue_w(q);
                issue_x(q, s);
            }
            if (++s == ns) s = 0, ++j;
            ++issued;
        }
        // the outlier slice: chunks of W16[o, this CTA's columns] and the X values
        const int cnt = (!WRITE_I32 && a.use_outliers && !a.w8) ? ldg_cg_s32(&a.hdr->outlier_count) : 0;
        const int nchunks = cnt > 0 ? (cnt + chunk - 1) / chunk : 0;
        for (int c = 0; c < nchunks && ok; ++c) {
            const int v = total + c;
            if (!(ok = wait_slot(v))) break;
            const int q = v % R, o0 = c * chunk, nc = min(chunk, cnt - o0);
            const int xb = (nc * 2 + 15) & ~15;  // X values of the chunk, rounded up to 16 bytes (zero-padded)
            uint8_t* dst = ring + (size_t)q * SB;
            if (leader) mbar_arrive_expect_tx(&sb.full[q], (uint32_t)(nc * seg + M * xb));
            __syncwarp();
            for (int o = lane; o < nc; o += 32) {
                const int k = ldg_cg_s32(a.outlier_idx + o0 + o);
                bulk_load_1d(dst + o * seg, a.W16 + (size_t)k * N + n_begin, (uint32_t)seg, &sb.full[q]);
            }
            for (int i = lane; i < M; i += 32)
                bulk_load_1d(dst + chunk * seg + i * kGsChunk * 2, a.xo + (size_t)i * a.xo_pitch + o0, (uint32_t)xb,
                             &sb.full[q]);
            ++issued;
        }
        // no copy may still target shared memory when the CTA ends: wait for the
        // last fill of every slot (already complete when the consumers finished)
        if (leader) {
            const int filled = min(R, issued);
            for (int sl = 0; sl < filled; ++sl) {
                const int last = sl + ((issued - 1 - sl) / R) * R;  // last stage that used slot sl
                mbar_wait_bounded(&sb.full[sl], (uint32_t)((last / R) & 1), 1u << 20, nullptr);
            }
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    auto wait_warp = [&](uint64_t* bar, uint32_t par, uint32_t where) -> bool {
        uint32_t got = 0;
        if (lane == 0) got = mbar_wait_bounded(bar, par, a.spin_limit, abort_flag) ? 1u : 0u;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got && lane == 0 && !*abort_flag) fail(32);
        return got != 0;
    };
    pdl_wait();  // the outlier count is written by the X pass
    const int cnt = (!WRITE_I32 && a.use_outliers) ? ldg_cg_s32(&a.hdr->outlier_count) : 0;
    const int nchunks = (cnt > 0 && !a.w8) ? (cnt + chunk - 1) / chunk : 0;

    int q = 0;
    uint32_t ph = 0;
    auto next_slot = [&]() {
        if (++q == R) q = 0, ph ^= 1u;
    };
    for (int j = 0; j < my_tiles; ++j) {
        // ---- int8 stages of tile j: partial sums of this thread
        int acc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};  // mma.sync fragments (MT tiles)
        int dacc[2] = {0, 0};                          // dp4a: rows 0, 1 of X
        for (int s = 0; s < ns; ++s) {
            if (!wait_warp(&sb.full[q], ph, 33)) return;
            const uint8_t* st = ring + (size_t)q * SB;
            const uint8_t* sx = st + kGsCols * SK;
            const int gs0 = s * NST;  // K step of local step 0
            if (MODE == kGsDp4a) {
                // warp pair (2p, 2p+1) takes local steps p, p+4, ...; thread: row n, 16-byte vector v
                const int n = 8 * (warp & 1) + (lane >> 2), v = lane & 3, pr = warp >> 1;
#pragma unroll 4
                for (int ls = pr; ls < NST; ls += 4) {
                    const int g = gs0 + ls;
                    const bool tl = p.tail && g == p.kfull;  // the ragged last step: from the tail area
                    if (g > p.kfull || (g == p.kfull && !tl) || (tl && 16 * v >= p.tail)) continue;
                    const uint4 w = *reinterpret_cast<const uint4*>(tl ? st + p.tail_off + n * 64 + 16 * v
                                                                       : st + ls * 1024 + n * 64 + 16 * v);
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        if (m < M) {
                            const uint4 x = *reinterpret_cast<const uint4*>(
                                tl ? st + p.tail_off + (kGsCols + m) * 64 + 16 * v : sx + ls * (M * 64) + m * 64 + 16 * v);
                            dacc[m] = __dp4a((int)w.x, (int)x.x, dacc[m]);
                            dacc[m] = __dp4a((int)w.y, (int)x.y, dacc[m]);
                            dacc[m] = __dp4a((int)w.z, (int)x.z, dacc[m]);
                            dacc[m] = __dp4a((int)w.w, (int)x.w, dacc[m]);
                        }
                    }
                }
            } else {
                // warp w takes local steps [w * NST/8, (w+1) * NST/8); thread (g, tq): weight rows
                // g and g+8 and X rows g (+8) at byte 16 tq of each step
                constexpr int MT = MODE == kGsMma2 ? 2 : 1;
                const int g = lane >> 2, tq = lane & 3;
                const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int x = 0; x < NST / kGsWarps; ++x) {
                    const int ls = warp * (NST / kGsWarps) + x, gk = gs0 + ls;
                    const bool tl = p.tail && gk == p.kfull;
                    const uint8_t* wb = tl ? st + p.tail_off : st + ls * 1024;
                    const uint4 w0 = *reinterpret_cast<const uint4*>(wb + g * 64 + 16 * tq);
                    const uint4 w1 = *reinterpret_cast<const uint4*>(wb + (g + 8) * 64 + 16 * tq);
                    // steps past K are zero in shared memory (box fill); the tail step is
                    // valid for its first p.tail bytes only
                    const bool kok = gk < p.kfull || (tl && 16 * tq < p.tail);
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        const int i = g + 8 * t;
                        const uint4 xf = (kok && i < M) ? *reinterpret_cast<const uint4*>(
                                                              tl ? st + p.tail_off + (kGsCols + i) * 64 + 16 * tq
                                                                 : sx + ls * (M * 64) + i * 64 + 16 * tq)
                                                        : z;
                        imma_16832(acc[t], w0.x, w1.x, w0.y, w1.y, xf.x, xf.y);
                        imma_16832(acc[t], w0.z, w1.z, w0.w, w1.w, xf.z, xf.w);
                    }
                }
            }
            __syncwarp();  // every lane has read the stage
            if (lane == 0) mbar_arrive(&sb.empty[q]);
            next_slot();
        }
        // ---- tile end: partial sums -> s_red; after the barrier, C of the tile -> s_c.
        // Passing red[j & 1] means every warp finished tile j - 1, so s_red[j & 1]
        // (last read at tile j - 2) is free.
        const int bb = j & 1;
        if (MODE == kGsDp4a) {
            // sum the four 16-byte vectors of a row, then one partial per warp pair
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                dacc[m] += __shfl_xor_sync(0xffffffffu, dacc[m], 1);
                dacc[m] += __shfl_xor_sync(0xffffffffu, dacc[m], 2);
            }
            if ((lane & 3) == 0) {
                const int n = 8 * (warp & 1) + (lane >> 2), pr = warp >> 1;
                s_red[bb][pr][0][n] = dacc[0];
                s_red[bb][pr][1][n] = dacc[1];
            }
        } else {
            // accumulator layout: d0,d1 -> (column g, x rows 8t+2q, +1); d2,d3 -> (column g+8, same rows)
            const int g = lane >> 2, tq = lane & 3;
#pragma unroll
            for (int t = 0; t < (MODE == kGsMma2 ? 2 : 1); ++t) {
                const int i0 = 8 * t + 2 * tq;
                s_red[bb][warp][i0][g] = acc[t][0];
                s_red[bb][warp][i0 + 1][g] = acc[t][1];
                s_red[bb][warp][i0][g + 8] = acc[t][2];
                s_red[bb][warp][i0 + 1][g + 8] = acc[t][3];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.red[bb]);
        if (!wait_warp(&sb.red[bb], (uint32_t)((j >> 1) & 1), 34)) return;
        {
            const int ri = tid >> 4, nl = tid & 15;
            if (ri < M) {
                int32_t c = 0;
#pragma unroll
                for (int w = 0; w < NPART; ++w) c += s_red[bb][w][ri][nl];
                s_c[(j * M + ri) * kGsCols + nl] = c;
            }
        }
    }
    // every warp's writes of s_c are done: one more pass of the tile barrier
    {
        const int bb = my_tiles & 1;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.red[bb]);
        if (!wait_warp(&sb.red[bb], (uint32_t)((my_tiles >> 1) & 1), 35)) return;
    }

    // ---- A4: the outlier slice over this CTA's columns, chunk by chunk from the ring
    const int nout = M * cols;  // outputs of this CTA, e -> (row e / cols, column e % cols)
    for (int c = 0; c < nchunks; ++c) {
        if (!wait_warp(&sb.full[q], ph, 36)) return;
        const uint8_t* st = ring + (size_t)q * SB;
        const int o0 = c * chunk, nc = min(chunk, cnt - o0);
        const __half* xv = reinterpret_cast<const __half*>(st + chunk * seg);
        for (int e = tid; e < nout; e += kGsWarps * 32) {
            const int ri = e / cols, col = e - ri * cols;
            float f = c == 0 ? 0.0f : s_f[e];
            for (int o = 0; o < nc; ++o)
                f = fmaf(elem_f<T>(xv[ri * kGsChunk + o]),
                         elem_f<T>(*reinterpret_cast<const __half*>(st + o * seg + col * 2)), f);
            s_f[e] = f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.empty[q]);
        next_slot();
    }

    // ---- A5: scales, the outlier slice, and the store (each thread its own outputs)
    for (int e = tid; e < nout; e += kGsWarps * 32) {
        const int ri = e / cols, col = e - ri * cols;
        const int jt = col >> 4, nl = col & 15;
        const int32_t cv = s_c[(jt * M + ri) * kGsCols + nl];
        const int n = n_begin + col;
        if (WRITE_I32) {
            reinterpret_cast<int32_t*>(a.out)[(size_t)ri * N + n] = cv;
            continue;
        }
        float f = nchunks > 0 ? s_f[e] : 0.0f;
        if (a.w8 && cnt > 0) {
            // int8 weight storage: outlier rows from the kept fp16 rows or the dequantized codes
            for (int o = 0; o < cnt; ++o) {
                const int k = __ldcg(a.outlier_idx + o);
                const __half x = __ldcg(a.xo + (size_t)ri * a.xo_pitch + o);
                f = fmaf(elem_f<T>(x), w16_value<T>(a, k, n), f);
            }
        }
        const float scale = __ldcg(a.row_scale + ri) * __ldg(a.col_scale + n) * (1.0f / 16129.0f);
        reinterpret_cast<uint16_t*>(a.out)[(size_t)ri * N + n] = Fmt<T>::from_float(fmaf((float)cv, scale, f));
    }
}

}  // namespace llmint8
