// Device-side helpers shared by the LLM.int8() kernels: workspace header, the
// device error word, bounded waits, and thin inline-PTX wrappers (mbarrier,
// TMA, tcgen05).  sm_103a only.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace llmint8 {

// ----------------------------------------------------------------------------
// Workspace header (first 256 bytes of every workspace)
// ----------------------------------------------------------------------------
struct WsHeader {
    uint32_t status;         // device error word: 0 or an llmint8_status value
    int32_t outlier_count;   // |O| of the last call
    uint32_t timeout_where;  // diagnostic: which wait gave up (role id)
    uint32_t pad[61];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

constexpr uint32_t kStatusTimeout = 5;  // == LLMINT8_ETIMEOUT

// Default poll budget of a bounded wait.  A healthy wait in these kernels ends
// within microseconds; 2^27 polls (each try_wait may suspend up to ~0.5 us) is
// far beyond that and still ends a stuck kernel in bounded time.
constexpr uint32_t kDefaultSpinLimit = 1u << 27;

__device__ __forceinline__ void record_error(WsHeader* h, uint32_t code, uint32_t where) {
    if (h) {
        atomicCAS(&h->status, 0u, code);
        atomicExch(&h->timeout_where, where);
    }
}

// ----------------------------------------------------------------------------
// Small numeric helpers
// ----------------------------------------------------------------------------

// Four int8 codes packed in a word -> two half2 holding the exact integer
// values.  Uses the fp16 bit pattern 0x6400 + u == 1024 + u for u in [0, 255]:
// flip the sign bits (u = q + 128), splice each byte under 0x64, subtract 1152.
__device__ __forceinline__ void s8x4_to_half2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(u), "r"(0x64646464u));
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    __half2 l = __hsub2(*reinterpret_cast<__half2*>(&lo), bias);
    __half2 h = __hsub2(*reinterpret_cast<__half2*>(&hi), bias);
    lo = *reinterpret_cast<uint32_t*>(&l);
    hi = *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// L2-coherent load (bypasses L1).  Used for every buffer an earlier kernel of
// the same call writes: with programmatic dependent launch the reading kernel is
// already running while that buffer is produced, so the non-coherent read-only
// path (ld.global.nc), whose data must not change during the reader's lifetime,
// is not allowed for it.
__device__ __forceinline__ uint4 ldg_cg_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
    return v;
}

// Streaming load that does not allocate in L1 (weights are read exactly once).
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Asynchronous 16-byte global -> shared copies (completion per thread via wait_all).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src);
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ----------------------------------------------------------------------------
// mbarrier
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}

// 16-bit element formats of X, W and Y: fp16 (__half) or bf16 (__nv_bfloat16).
// Wherever no arithmetic touches them the values are moved as raw 16-bit words
// (held in __half-typed storage); Fmt<T> converts at the few places that compute.
template <typename T>
struct Fmt;
template <>
struct Fmt<__half> {
    static constexpr bool kBF16 = false;
    __device__ __forceinline__ static float2 to_float2(uint32_t w) {
        return __half22float2(*reinterpret_cast<const __half2*>(&w));
    }
    __device__ __forceinline__ static float to_float(uint16_t b) { return __half2float(__ushort_as_half(b)); }
    __device__ __forceinline__ static uint16_t from_float(float f) { return __half_as_ushort(__float2half_rn(f)); }
    __device__ __forceinline__ static uint32_t pack2(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
};
template <>
struct Fmt<__nv_bfloat16> {  // bf16 = the upper half of a binary32
    static constexpr bool kBF16 = true;
    __device__ __forceinline__ static float2 to_float2(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    __device__ __forceinline__ static float to_float(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
    __device__ __forceinline__ static uint16_t from_float(float f) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(f));
    }
    __device__ __forceinline__ static uint32_t pack2(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
};
// the value of a raw 16-bit word of format T
template <typename T>
__device__ __forceinline__ float elem_f(__half raw) {
    return Fmt<T>::to_float(__half_as_ushort(raw));
}

// A4 weight without a full fp16 copy of W: code q of a column whose absmax is
// s_w, dequantized as RNE_T(fp32(q) * fp32(s_w / 127)), each step rounded to
// nearest even (a code times its scale, the scale stored as the absmax); the
// raw 16-bit word of format T.
template <typename T>
__device__ __forceinline__ __half dequant_weight(int8_t q, float s_w) {
    return __ushort_as_half(Fmt<T>::from_float(__fmul_rn((float)q, __fdiv_rn(s_w, 127.0f))));
}

// Hint: bring [p, p + bytes) into L2 (p 16-byte aligned, bytes a multiple of 16).
// It moves nothing into the SM, so it may precede griddepcontrol.wait even for
// data the predecessor writes: every read after the wait goes through L2, which
// also receives those writes.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// 32-bit load through L2, kept in program order (issued where it is written, so
// independent loads go out together).
__device__ __forceinline__ int ldg_cg_s32(const int* p) {
    int v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on a barrier phase.  Returns false (and the caller must bail
// out) when the poll budget is exhausted or, if abort_flag is given, when
// another thread of the CTA has flagged an abort.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit,
                                                  volatile uint32_t* abort_flag) {
    for (uint32_t i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort_flag != nullptr && (i & 1023u) == 1023u && *abort_flag) return false;
    }
    return false;
}

// ----------------------------------------------------------------------------
// Bulk (non-tensor) async copies between global and shared memory.  Both
// addresses 16-byte aligned, size a multiple of 16.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void bulk_load_1d(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_store_1d(void* gmem_dst, const void* smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// at most N of this thread's committed bulk store groups still reading shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// all of this thread's committed bulk store groups complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Orders this thread's generic-proxy writes to shared memory before later
// async-proxy reads of it (a bulk store of data written with st.shared).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) -- 2D tiled loads into shared memory
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const void* desc) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(desc) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* desc, uint64_t* bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(desc), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// 2D tiled store of a shared-memory box (laid out as the tensor map's swizzle
// says) to global memory; completes in this thread's current bulk group.
// Elements of the box outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const void* desc, const void* smem_src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(desc),
                 "r"(smem_u32(smem_src)), "r"(x), "r"(y)
                 : "memory");
}

// ----------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core, TMEM accumulators)
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_result, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (fp16 inputs, fp32 accumulate).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on an mbarrier once all previously issued tcgen05.mma of this thread completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// ---- CTA pairs (cluster of two): tcgen05 with .cta_group::2 ----------------
// One MMA, issued by a thread of the first CTA, multiplies the A rows held by
// both CTAs (128 each, same shared-memory offset) by the B columns held by both
// (N/2 each) and accumulates rows 0..127 in the first CTA's TMEM and 128..255 in
// the second's.  Allocation is collective: one warp of each CTA issues it, and
// the same columns are allocated in both.  Every tcgen05 instruction of a
// kernel that uses pairs carries .cta_group::2.
__device__ __forceinline__ uint32_t cluster_cta_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of the variable at shared address `addr` in CTA `rank`
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
// TMA tile load into this CTA's shared memory whose completion is signalled on
// an mbarrier that may sit in the peer CTA (shared::cluster address)
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const void* desc, uint32_t bar_cluster, int x,
                                                 int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(desc), "r"(bar_cluster), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* smem_result, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on the mbarrier at this offset in every CTA of `cta_mask` once all
// previously issued tcgen05.mma of this thread completed
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp gets lane
// (base lane + t), columns [col, col+32).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand tile whose rows are
// 128 bytes (64 fp16) and which TMA wrote with 128-byte swizzling: 8-row
// groups are 1024 bytes apart (stride byte offset); the leading byte offset is
// unused for swizzled K-major layouts (set to 1); bits 46-47 hold the
// descriptor version 1; bits 61-63 select the 128-byte swizzle (value 2).
__device__ __forceinline__ uint64_t make_sdesc_k128(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)1u << 16;                    // LBO (unused)
    d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;  // SBO = 1024 B
    d |= (uint64_t)1u << 46;                    // version
    d |= (uint64_t)2u << 61;                    // SWIZZLE_128B
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: fp16 (or, with bf16, bf16)
// A and B, fp32 D, both operands K-major, shape M x N.
__host__ __device__ constexpr uint32_t make_idesc_f16(int M, int N, bool bf16 = false) {
    return (1u << 4)                          // D format: f32
           | ((bf16 ? 1u : 0u) << 7)          // A format: f16 (0) or bf16 (1)
           | ((bf16 ? 1u : 0u) << 10)         // B format: f16 (0) or bf16 (1)
           | (0u << 15) | (0u << 16)          // A, B K-major
           | ((uint32_t)(N >> 3) << 17)       // N / 8
           | ((uint32_t)(M >> 4) << 24);      // M / 16
}

}  // namespace llmint8
