// rmsq_device.cuh -- device code of the fused residual-add + RMSNorm + FP8 / NVFP4 / MXFP4 kernels
// for sm_103a (GB300).
//
// One kernel template covers every mode, input type and schedule. A row processor (a CTA, a warp
// or a cluster) owns whole rows: its threads split a row into 16-byte vectors (vector v goes to
// thread v % T, so a warp touches 512 contiguous bytes per step), add the residual, reduce the
// sum of squares, form y = s * rstd * (gamma + offset) and quantise. The row is read from HBM
// exactly once.
//
// Four schedules fetch the row:
//   SCHED_PIPE  persistent CTAs with a ring of `stages` shared-memory row buffers filled by the
//               TMA bulk-copy engine (cp.async.bulk + mbarrier transaction counts). Thread 0
//               refills a buffer with the CTA's next row as soon as the CTA has read it, so
//               several rows per SM stay in flight while the CTA computes. Rows are dealt out
//               round-robin, the last quarter one at a time from a per-launch counter.
//   SCHED_REG   persistent CTAs that load their row straight into registers with 128-bit
//               streaming loads; latency is hidden by the other CTAs on the SM.
//   SCHED_WARP  row per warp, for short rows: every warp of a CTA owns whole rows with its own
//               ring of row buffers and mbarriers (lane 0 issues the bulk copies), and all
//               reductions are warp shuffles -- no CTA barrier and no cross-warp stage per row.
//   SCHED_CLUSTER  rows wider than one CTA's ring holds: a thread-block cluster of C CTAs
//               shares each row, CTA k taking the k-th 1/C of it through its own ring. The
//               CTAs' row sums (and maxima) meet in distributed shared memory: each CTA writes
//               its partial into its own exchange slot, one cluster barrier, then every CTA
//               reads all C slots in rank order, so every CTA forms the same totals.
//
// Method sources: Modular Mojo API docs "rms_norm_fused_fp8" / "allreduce_residual_rmsnorm_fp8"
// (FP8 row scale with scale_ub, residual_output, weight_offset on gamma) and FlashInfer
// "cute_dsl/rmsnorm_fp4quant.py" (RMSNormFP4QuantKernel phases 2-3: rstd, block amax, E4M3 /
// UE8M0 block scale, E2M1 packing, swizzled 128x4 scale layout).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace rmsq {

enum { DT_BF16 = 0, DT_FP16 = 1, DT_F32 = 2 };
// MODE_AMAX is the NVFP4 global-scale pre-pass: y is formed but only max |y| leaves the kernel.
enum { MODE_FP8 = 0, MODE_NVFP4 = 1, MODE_MXFP4 = 2, MODE_AMAX = 3 };
enum { SCHED_PIPE = 1, SCHED_REG = 2, SCHED_WARP = 3, SCHED_CLUSTER = 4 };

// Error flag bits set on the device.
// ERRF_DRAIN_TIMEOUT: after a timed-out wait, a CTA's wait for its own copies in flight also ran
// out, so it may have exited while a copy into its shared memory was still outstanding.
enum { ERRF_WAIT_TIMEOUT = 1u, ERRF_DRAIN_TIMEOUT = 2u };

struct Params {
    const void* x;            // [rows x hidden]
    const void* res;          // [rows x hidden] or null
    void* res_out;            // [rows x hidden] or null
    const void* gamma;        // [hidden]
    void* out;                // codes
    void* scale_out;          // FP8 row scales / FP4 block scales
    const float* gs;          // NVFP4 global scale (device)
    unsigned int* err;        // device error word
    long long rows;
    int nvec;                 // 16-byte vectors per row
    int hidden;
    float eps;
    float offset;
    float scale_ub;
    int scale_dtype;          // FP8: DT_F32 / DT_BF16 / DT_FP16
    int swizzled;             // FP4: swizzled 128x4 scale layout
    int nsf;                  // FP4: block scales per row
    int k_tiles;              // FP4 swizzled: 4-scale tiles per row
    int stages;               // SCHED_PIPE / SCHED_WARP: ring depth (per ring)
    unsigned long long timeout_ns;
    // Ring schedules: rows below rows_static go round-robin over the row processors (CTAs, or
    // warps for SCHED_WARP); the rest are handed out one at a time from the counter *rowctr,
    // which starts at 0 and is left at 0. rowctr may be null, with rows_static = rows.
    unsigned int* rowctr;
    long long rows_static;
    // MODE_AMAX: two words of the launch's scratch slot, both 0 at launch and left at 0: [0] the
    // running max |y| (bits), [1] the count of CTAs done. The last CTA turns the max into gs.
    unsigned int* amax_slot;
};

// ------------------------------------------------------------------------------------------
// PTX helpers (hand-written): mbarrier, bulk copy, timers, conversions
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before later async-proxy
// (bulk copy) accesses to the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Completes the barrier's phase without a copy (count 1): the slot carries no row.
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Thread-block cluster: this CTA's rank, the cluster size, this cluster's index and the count.
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size()
{
    uint32_t r;
    asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id()
{
    uint32_t r;
    asm("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_count()
{
    uint32_t r;
    asm("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster: shared-memory writes before it are visible to the
// cluster's reads after it.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// The two halves of cluster_sync, for work placed between them. Every thread of every CTA calls
// them alternately, arrive first. A thread whose earlier writes some other CTA reads after the
// barrier arrives with release semantics (publish); any other thread arrives relaxed, without the
// memory fence.
__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void cluster_arrive_as(bool publish)
{
    if (publish) asm volatile("barrier.cluster.arrive.release;" ::: "memory");
    else asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}

// Read a float4 at shared address `addr` of the CTA with cluster rank `rank`.
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr, uint32_t rank)
{
    uint32_t raddr;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(addr), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(raddr)
                 : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long globaltimer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the given phase of an mbarrier, for at most timeout_ns. Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long timeout_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
}

// L2 priority of the row loads. Normal priority (rather than evict-first) lets the kernel's own
// dirty output lines leave L2 while it runs instead of piling up until it ends: measured on
// GB300, the ncu DRAM throughput of the NVFP4 / MXFP4 launches rises by 3-4 points and the long
// MXFP4 launches get 3 % shorter.
__device__ __forceinline__ uint64_t l2_evict_normal_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Global -> shared bulk copy (TMA engine), completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint4 ld_stream_v4(const uint4* p)
{
    uint4 v;
    asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_v4(void* p, uint4 v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_v2(void* p, uint32_t a, uint32_t b)
{
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void st_u32(void* p, uint32_t a)
{
    asm volatile("st.global.u32 [%0], %1;" ::"l"(p), "r"(a) : "memory");
}

__device__ __forceinline__ void st_u16(void* p, uint16_t a)
{
    asm volatile("st.global.u16 [%0], %1;" ::"l"(p), "h"(a) : "memory");
}

// Two fp32 -> two E4M3 codes (round to nearest even, satfinite); `lo` lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Eight fp32 -> eight E2M1 codes packed in a u32 (RNE, satfinite); element j in nibble j.
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float (&v)[8])
{
    uint32_t r;
    asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
        "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
        : "=r"(r)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

// Four fp32 -> four E2M1 codes in the low 16 bits.
__device__ __forceinline__ uint32_t cvt_e2m1x4(const float (&v)[4])
{
    uint32_t r;
    asm("{\n\t.reg .b8 q0, q1;\n\t.reg .b16 h;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
        "mov.b16 h, {q0, q1};\n\t"
        "cvt.u32.u16 %0, h;\n\t}"
        : "=r"(r)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]));
    return r;
}

// Exact value of an E4M3 code (hardware e4m3 -> f16 conversion is exact, subnormals included).
__device__ __forceinline__ float e4m3_value(uint32_t code)
{
    uint32_t h2;
    const uint16_t c = static_cast<uint16_t>(code & 0xFFu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    float f;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, l;\n\t}" : "=f"(f) : "r"(h2));
    return f;
}

// ------------------------------------------------------------------------------------------
// Element types: 16-byte vectors of bf16 / fp16 (8 elements) or fp32 (4 elements)
// ------------------------------------------------------------------------------------------

template <int DT> struct Elem;

template <> struct Elem<DT_BF16> {
    static constexpr int EPV = 8;
    // Exact products of the two bf16 halves of a and b (mixed-precision FMA with a zero addend:
    // a 16-bit by 16-bit product is exact in fp32).
    static __device__ __forceinline__ float2 mul_halves(uint32_t a, uint32_t b)
    {
        float2 r;
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %3;\n\t"
            "fma.rn.f32.bf16 %0, a0, b0, 0f80000000;\n\tfma.rn.f32.bf16 %1, a1, b1, 0f80000000;\n\t}"
            : "=f"(r.x), "=f"(r.y)
            : "r"(a), "r"(b));
        return r;
    }
    // acc + (halves of a)^2, one rounding each.
    static __device__ __forceinline__ float2 sq_acc(uint32_t a, float2 acc)
    {
        float2 r;
        asm("{\n\t.reg .b16 a0, a1;\n\tmov.b32 {a0, a1}, %2;\n\t"
            "fma.rn.f32.bf16 %0, a0, a0, %3;\n\tfma.rn.f32.bf16 %1, a1, a1, %4;\n\t}"
            : "=f"(r.x), "=f"(r.y)
            : "r"(a), "f"(acc.x), "f"(acc.y));
        return r;
    }
    // Element pairs (2j, 2j+1) as float2, exact.
    static __device__ __forceinline__ void pairs(const uint4& v, float2 (&f)[4])
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
    }
    static __device__ __forceinline__ void unpack(const uint4& v, float (&f)[8])
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    // Correctly rounded bf16 sums (add.rn.bf16x2).
    static __device__ __forceinline__ uint4 add(const uint4& a, const uint4& b)
    {
        uint4 r;
        asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r.x) : "r"(a.x), "r"(b.x));
        asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r.y) : "r"(a.y), "r"(b.y));
        asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r.z) : "r"(a.z), "r"(b.z));
        asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r.w) : "r"(a.w), "r"(b.w));
        return r;
    }
};

template <> struct Elem<DT_FP16> {
    static constexpr int EPV = 8;
    static __device__ __forceinline__ float2 mul_halves(uint32_t a, uint32_t b)
    {
        float2 r;
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %3;\n\t"
            "fma.rn.f32.f16 %0, a0, b0, 0f80000000;\n\tfma.rn.f32.f16 %1, a1, b1, 0f80000000;\n\t}"
            : "=f"(r.x), "=f"(r.y)
            : "r"(a), "r"(b));
        return r;
    }
    static __device__ __forceinline__ float2 sq_acc(uint32_t a, float2 acc)
    {
        float2 r;
        asm("{\n\t.reg .b16 a0, a1;\n\tmov.b32 {a0, a1}, %2;\n\t"
            "fma.rn.f32.f16 %0, a0, a0, %3;\n\tfma.rn.f32.f16 %1, a1, a1, %4;\n\t}"
            : "=f"(r.x), "=f"(r.y)
            : "r"(a), "f"(acc.x), "f"(acc.y));
        return r;
    }
    static __device__ __forceinline__ void pairs(const uint4& v, float2 (&f)[4])
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float lo, hi;
            asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
                "cvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
                : "=f"(lo), "=f"(hi)
                : "r"(w[i]));
            f[i] = make_float2(lo, hi);
        }
    }
    static __device__ __forceinline__ void unpack(const uint4& v, float (&f)[8])
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float lo, hi;
            asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
                "cvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
                : "=f"(lo), "=f"(hi)
                : "r"(w[i]));
            f[2 * i] = lo;
            f[2 * i + 1] = hi;
        }
    }
    static __device__ __forceinline__ uint4 add(const uint4& a, const uint4& b)
    {
        uint4 r;
        asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r.x) : "r"(a.x), "r"(b.x));
        asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r.y) : "r"(a.y), "r"(b.y));
        asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r.z) : "r"(a.z), "r"(b.z));
        asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r.w) : "r"(a.w), "r"(b.w));
        return r;
    }
};

template <> struct Elem<DT_F32> {
    static constexpr int EPV = 4;
    // (not used: fp32 rows always take the unpacked path)
    static __device__ __forceinline__ float2 mul_halves(uint32_t, uint32_t) { return make_float2(0.f, 0.f); }
    static __device__ __forceinline__ float2 sq_acc(uint32_t, float2 acc) { return acc; }
    static __device__ __forceinline__ void pairs(const uint4& v, float2 (&f)[2])
    {
        f[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
        f[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
    }
    static __device__ __forceinline__ void unpack(const uint4& v, float (&f)[4])
    {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    static __device__ __forceinline__ uint4 add(const uint4& a, const uint4& b)
    {
        uint4 r;
        r.x = __float_as_uint(__fadd_rn(__uint_as_float(a.x), __uint_as_float(b.x)));
        r.y = __float_as_uint(__fadd_rn(__uint_as_float(a.y), __uint_as_float(b.y)));
        r.z = __float_as_uint(__fadd_rn(__uint_as_float(a.z), __uint_as_float(b.z)));
        r.w = __float_as_uint(__fadd_rn(__uint_as_float(a.w), __uint_as_float(b.w)));
        return r;
    }
};

// Packed fp32 pairs (Blackwell f32x2 instructions: two IEEE round-to-nearest operations per
// instruction), through CUDA's float2 intrinsics so the compiler can keep pairs in register pairs.
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }

__device__ __forceinline__ float2 sub2(float2 a, float2 b)
{
    return __fadd2_rn(a, make_float2(-b.x, -b.y));
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

__device__ __forceinline__ float max3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float2 splat(float v) { return make_float2(v, v); }

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// max |v| over the 32 lanes of a full warp, in one warp-wide reduction instruction (every lane
// gets the result). For the non-negative finite values the kernels reduce, it equals warp_max.
__device__ __forceinline__ float warp_max_abs(float v)
{
    float r;
    asm volatile("redux.sync.max.abs.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

// UE8M0 code of a block with max |y| = a >= 0: the smallest e with 6 * 2^e >= a, plus 127,
// clamped to [0, 255]; 0 for a = 0. Exact, from a's bits: for a = m * 2^E with m in [1, 2),
// a / 6 <= 2^(E-2) exactly when m <= 1.5, so e = E - 2 if m <= 1.5 and E - 1 otherwise.
// Subnormal a (< 2^-126) gives e <= -128, hence code 0.
__device__ __forceinline__ uint32_t ue8m0_code(float a)
{
    const uint32_t bits = __float_as_uint(a);
    const int biased = static_cast<int>(bits >> 23);          // a >= 0: no sign bit
    if (biased == 0) return 0u;                                // zero or subnormal
    const int e = biased - 127 - 2 + ((bits & 0x7FFFFFu) > 0x400000u ? 1 : 0);
    int code = e + 127;
    code = code < 0 ? 0 : (code > 255 ? 255 : code);
    return static_cast<uint32_t>(code);
}

// 2^(127 - code) for code in [1, 254] (exact), 0 for code 0.
__device__ __forceinline__ float ue8m0_inv_factor(uint32_t code)
{
    return code == 0u ? 0.0f : __uint_as_float((254u - code) << 23);
}

// ------------------------------------------------------------------------------------------
// Exactly rounded row math (FP8)
//
// FP8 codes are decided by comparing y / scale with rounding boundaries. With 16-bit inputs,
// y_i / scale = 448 * (s_i w_i) / (s_m w_m) in exact arithmetic (rstd cancels): a ratio of short
// numbers that lands on a boundary far more often than random data would, so the way such a
// near-tie goes is decided by the fp32 roundings of rstd, y and the scale. The FP8 kernel
// therefore forms rstd, y and the scale as the correctly rounded fp32 values of their definitions
// and rounds the exact quotient y / scale to E4M3:
//   sum of squares  compensated (TwoSum) fp32 accumulation: hi + lo within ~2^-45 of the exact sum
//   rstd            RN(1 / sqrt(sum / H + eps)) from one Newton step in float-float arithmetic
//   y               RN(s * w * rstd) with s * w split exactly by an FMA
//   y / scale       the correctly rounded fp32 quotient; when it lands exactly on an E4M3
//                   boundary while the exact quotient does not (found from the exact remainder),
//                   it moves one unit toward the exact value, so the E4M3 RNE conversion rounds
//                   the exact quotient
// FP4 codes see no such cancellation (the block scale is itself rounded, or a power of two applied
// to y exactly), so the FP4 kernels and the amax pre-pass use a plain fp32 sum of squares and the
// correctly rounded rsqrt of the rounded mean.
// ------------------------------------------------------------------------------------------

struct FF {
    float hi, lo;
};

// a + b = s.hi + s.lo exactly (TwoSum; no ordering assumption).
__device__ __forceinline__ FF two_sum(float a, float b)
{
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return FF{s, e};
}

__device__ __forceinline__ FF ff_add(FF a, FF b)
{
    FF s = two_sum(a.hi, b.hi);
    s.lo = __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo));
    return s;
}

// TwoSum on two independent lanes.
__device__ __forceinline__ void two_sum2(float2 a, float2 b, float2& s, float2& e)
{
    s = add2(a, b);
    const float2 bb = sub2(s, a);
    e = add2(sub2(a, sub2(s, bb)), sub2(b, bb));
}

// a + b for non-negative a.hi, b.hi (partial sums of squares): Fast2Sum on the larger and the
// smaller high part gives the same exact split as TwoSum in fewer dependent steps.
__device__ __forceinline__ FF ff_add_pos(FF a, FF b)
{
    const float big = fmaxf(a.hi, b.hi), small = fminf(a.hi, b.hi);
    const float s = __fadd_rn(big, small);
    const float e = __fsub_rn(small, __fsub_rn(s, big));
    return FF{s, __fadd_rn(__fadd_rn(a.lo, b.lo), e)};
}

__device__ __forceinline__ FF shfl_xor_ff(FF v, int o)
{
    return FF{__shfl_xor_sync(0xFFFFFFFFu, v.hi, o), __shfl_xor_sync(0xFFFFFFFFu, v.lo, o)};
}

// RN_fp32(1 / sqrt(ss / H + eps)) for ss = hi + lo.
__device__ __forceinline__ float rstd_from_sum(FF ss, float H, float eps)
{
    const float q = __fdiv_rn(ss.hi, H);
    const float rem = fmaf(-q, H, ss.hi);                     // exact remainder of the division
    const float q_lo = __fdiv_rn(__fadd_rn(rem, ss.lo), H);
    FF m = two_sum(q, eps);
    m.lo = __fadd_rn(m.lo, q_lo);
    if (!(m.hi > 0.0f)) return __int_as_float(0x7F800000);    // 1 / sqrt(0)
    const float r0 = rsqrtf(m.hi);
    const float p_hi = __fmul_rn(r0, r0);
    const float p_lo = fmaf(r0, r0, -p_hi);
    const float t_hi = __fmul_rn(m.hi, p_hi);
    const float t_lo = __fadd_rn(fmaf(m.hi, p_hi, -t_hi), fmaf(m.hi, p_lo, __fmul_rn(m.lo, p_hi)));
    const float e = __fsub_rn(__fsub_rn(1.0f, t_hi), t_lo);   // 1 - m r0^2, t_hi ~ 1 so exact
    return __fadd_rn(r0, __fmul_rn(__fmul_rn(r0, 0.5f), e));
}

// As rstd_from_sum for a power-of-two H (inv_h = 1 / H exactly, so the mean is exact).
__device__ __forceinline__ float rstd_from_sum_pow2(FF ss, float inv_h, float eps)
{
    FF m = two_sum(__fmul_rn(ss.hi, inv_h), eps);
    m.lo = __fadd_rn(m.lo, __fmul_rn(ss.lo, inv_h));
    if (!(m.hi > 0.0f)) return __int_as_float(0x7F800000);
    const float r0 = rsqrtf(m.hi);
    const float p_hi = __fmul_rn(r0, r0);
    const float p_lo = fmaf(r0, r0, -p_hi);
    const float t_hi = __fmul_rn(m.hi, p_hi);
    const float t_lo = __fadd_rn(fmaf(m.hi, p_hi, -t_hi), fmaf(m.hi, p_lo, __fmul_rn(m.lo, p_hi)));
    const float e = __fsub_rn(__fsub_rn(1.0f, t_hi), t_lo);
    return __fadd_rn(r0, __fmul_rn(__fmul_rn(r0, 0.5f), e));
}

// RN(s * w * rstd) on a pair: s * w = hi + lo exactly, then one rounding of hi rstd + lo rstd.
__device__ __forceinline__ float2 norm_mul2(float2 s, float2 w, float2 rstd)
{
    const float2 hi = mul2(s, w);
    const float2 lo = fma2(s, w, make_float2(-hi.x, -hi.y));
    return fma2(hi, rstd, mul2(lo, rstd));
}

// RN(y / d) on a pair from inv = RN(1 / d) and nd = -d: one correction with the exact
// remainder y - q0 d.
__device__ __forceinline__ float2 div_rn2(float2 y, float2 nd, float2 inv)
{
    const float2 q0 = mul2(y, inv);
    return fma2(fma2(q0, nd, y), inv, q0);
}

// The correctly rounded fp32 quotient q can sit exactly on an E4M3 rounding boundary
// (1.xxx1 x 2^e: the low 19 mantissa bits zero and bit 19 set) while the exact quotient lies just
// off it; the E4M3 conversion would then break the tie to even instead of rounding the exact
// value. tie_key is zero exactly for such candidates.
__device__ __forceinline__ uint32_t tie_key(float q)
{
    return (__float_as_uint(q) & 0xFFFFFu) ^ 0x80000u;
}

// For a candidate, move q one unit toward the exact quotient y / d when the division was inexact,
// so the E4M3 conversion rounds the exact value. nd = -d.
__device__ __forceinline__ float untie(float q, float y, float nd)
{
    const float r = fmaf(q, nd, y);                          // y - q d, exact
    if (tie_key(q) != 0u || r == 0.0f) return q;
    const uint32_t b = __float_as_uint(q);
    const bool away = ((__float_as_uint(r) ^ b) >> 31) == 0u;  // |y / d| > |q|
    return __uint_as_float(away ? b + 1u : b - 1u);
}

// max |v| over the pairs of one vector, as a shallow tree.
template <int NP>
__device__ __forceinline__ float absmax_pairs(const float2 (&v)[NP])
{
    if constexpr (NP == 4) {
        return max3(max3(fabsf(v[0].x), fabsf(v[0].y), fabsf(v[1].x)),
                    max3(fabsf(v[1].y), fabsf(v[2].x), fabsf(v[2].y)),
                    fmaxf(fabsf(v[3].x), fabsf(v[3].y)));
    } else {
        return max3(fabsf(v[0].x), fabsf(v[0].y), fmaxf(fabsf(v[1].x), fabsf(v[1].y)));
    }
}

// w = fp32(gamma) + fp32(weight_offset) for this thread's vectors of the row. With up to four
// vectors per thread w is kept as fp32 pairs for the CTA's lifetime; with more, gamma stays
// packed and the offset is added per use.
template <class E, int VPT, bool UNPACKED = (VPT <= 4)>
struct GammaRegs;

template <class E, int VPT>
struct GammaRegs<E, VPT, true> {
    static constexpr int NP = E::EPV / 2;
    float2 w[VPT][NP];
    // group > 1: blocked order, slot k holds vector group * (tid + (k / group) * T) + k % group
    __device__ __forceinline__ void load(const uint4* gp, int tid, int T, int nv, float2 off,
                                         int group = 1)
    {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = group == 1 ? tid + k * T : group * (tid + (k / group) * T) + k % group;
            const uint4 gv = v < nv ? __ldg(gp + v) : make_uint4(0, 0, 0, 0);
            float2 f[NP];
            E::pairs(gv, f);
#pragma unroll
            for (int j = 0; j < NP; ++j) w[k][j] = add2(f[j], off);
        }
    }
    __device__ __forceinline__ void get(int k, float2 (&out)[NP]) const
    {
#pragma unroll
        for (int j = 0; j < NP; ++j) out[j] = w[k][j];
    }
};

template <class E, int VPT>
struct GammaRegs<E, VPT, false> {
    static constexpr int NP = E::EPV / 2;
    uint4 g[VPT];
    float2 off;
    __device__ __forceinline__ void load(const uint4* gp, int tid, int T, int nv, float2 o,
                                         int group = 1)
    {
        off = o;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = group == 1 ? tid + k * T : group * (tid + (k / group) * T) + k % group;
            g[k] = v < nv ? __ldg(gp + v) : make_uint4(0, 0, 0, 0);
        }
    }
    __device__ __forceinline__ void get(int k, float2 (&out)[NP]) const
    {
        E::pairs(g[k], out);
#pragma unroll
        for (int j = 0; j < NP; ++j) out[j] = add2(out[j], off);
    }
    // the 16-byte gamma vector k, as stored
    __device__ __forceinline__ uint4 packed(int k) const { return g[k]; }
};

// w for the FP8 kernels with a weight offset and 16-bit input: no registers held across the
// row. Each use re-reads the thread's gamma vector (16 KB at most for a row of 8192, resident in
// L1 for the kernel's lifetime) and adds the offset; those kernels use w once per row, and the
// registers saved let three 256-thread CTAs share an SM.
template <class E, int VPT>
struct GammaL1 {
    static constexpr int NP = E::EPV / 2;
    const uint4* gp;
    int tid, T, nv;
    float2 off;
    __device__ __forceinline__ void load(const uint4* g, int t, int TT, int n, float2 o, int = 1)
    {
        gp = g;
        tid = t;
        T = TT;
        nv = n;
        off = o;
    }
    __device__ __forceinline__ void get(int k, float2 (&out)[NP]) const
    {
        const int v = tid + k * T;
        E::pairs(v < nv ? __ldg(gp + v) : make_uint4(0, 0, 0, 0), out);
#pragma unroll
        for (int j = 0; j < NP; ++j) out[j] = add2(out[j], off);
    }
};

// w for the same kernels on the CTA-per-row ring, kept in shared memory as fp32 and formed once
// per CTA: two planes of 16 bytes per vector (pairs 0-1, then pairs 2-3), so a warp's reads of
// either plane are contiguous. The planner pays for the table with ring slots (one slot for rows
// of 8192: measured on GB300, 138.9 us against 144.0 us with w re-read from L1 and two slots).

template <class E, int VPT>
struct GammaSmem {
    static constexpr int NP = E::EPV / 2;
    uint32_t base;
    int tid, T, nv;
    __device__ __forceinline__ void init(uint32_t tab, const uint4* gp, int t, int TT, int n, float2 off)
    {
        base = tab;
        tid = t;
        T = TT;
        nv = n;
        for (int v = t; v < n; v += TT) {
            float2 f[NP];
            E::pairs(__ldg(gp + v), f);
#pragma unroll
            for (int j = 0; j < NP; ++j) f[j] = add2(f[j], off);
            st_shared_v4(base + v * 16u, make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y),
                                                    __float_as_uint(f[1].x), __float_as_uint(f[1].y)));
            st_shared_v4(base + (n + v) * 16u, make_uint4(__float_as_uint(f[2].x), __float_as_uint(f[2].y),
                                                          __float_as_uint(f[3].x), __float_as_uint(f[3].y)));
        }
    }
    __device__ __forceinline__ void load(const uint4*, int, int, int, float2, int = 1) {}
    __device__ __forceinline__ void get(int k, float2 (&out)[NP]) const
    {
        const int v = tid + k * T;
        uint4 a = make_uint4(0, 0, 0, 0), b = a;
        if (v < nv) {
            a = ld_shared_v4(base + v * 16u);
            b = ld_shared_v4(base + (nv + v) * 16u);
        }
        out[0] = make_float2(__uint_as_float(a.x), __uint_as_float(a.y));
        out[1] = make_float2(__uint_as_float(a.z), __uint_as_float(a.w));
        out[2] = make_float2(__uint_as_float(b.x), __uint_as_float(b.y));
        out[3] = make_float2(__uint_as_float(b.z), __uint_as_float(b.w));
    }
};

// Shared memory after the stage rings: [2][32] float2 sum-of-squares partials, [2][32] row
// maxima, [128] NVFP4 element factors gs / dec(s) indexed by the E4M3 block-scale code (the
// row-per-warp schedule reduces in registers and keeps only the factor table), then per ring
// [stages] mbarriers and [stages] row numbers of the slots, then (SCHED_CLUSTER) the cluster
// exchange slots: [3] float4 {sum hi, sum lo, max, stop}, used in turn, and [2] float4
// {amax, -, -, -}, or (FP8 with a weight offset on the CTA-per-row ring) the GammaSmem table of w.
constexpr int kRedFloats = 2 * 32 * 2 + 2 * 32 + 128;
constexpr int kRedFloatsWarp = 128;
constexpr int kClusterXchBytes = 5 * 16;

// ------------------------------------------------------------------------------------------
// The kernel
// ------------------------------------------------------------------------------------------

// The FP8 kernels with a weight offset and 16-bit input hold y in registers between the two
// row reductions (four vectors per thread) and take w from a shared-memory table (GammaSmem, on
// the CTA-per-row ring) or re-read gamma from L1 (GammaL1, the other schedules).
template <int DT, int MODE, int VPT, int SCHED, bool W16>
__host__ __device__ constexpr bool fp8_offset16()
{
    return MODE == MODE_FP8 && !W16 && DT != DT_F32 && VPT == 4 && SCHED != SCHED_CLUSTER;
}

// Registers per thread: those kernels, and the cluster-schedule kernels of 16-bit rows with a
// residual and four vectors per thread, are capped at 80 so that three CTAs of 256 threads fit
// an SM (the cap costs no spills there); the rest take what 512 threads allow.
template <int DT, bool RES, int MODE, int VPT, int SCHED, bool W16>
__host__ __device__ constexpr int reg_cap()
{
    return fp8_offset16<DT, MODE, VPT, SCHED, W16>() || (SCHED == SCHED_CLUSTER && RES && W16 && VPT == 4)
               ? 80
               : 128;
}

// W16: 16-bit input with weight_offset 0, so w = gamma is a 16-bit value and s * w, s^2 are
// exact products formed straight from packed halves by mixed-precision FMA (no unpacking).
template <int DT, bool RES, int MODE, int VPT, int SCHED, bool W16>
__global__ void __launch_bounds__(512, 1) __maxnreg__((reg_cap<DT, RES, MODE, VPT, SCHED, W16>()))
rmsq_row_kernel(const Params p)
{
    using E = Elem<DT>;
    constexpr int EPV = E::EPV;
    constexpr int NP = EPV / 2;                                      // element pairs per vector
    constexpr int BLOCK = MODE == MODE_NVFP4 ? 16 : 32;             // FP4 scale block
    constexpr int GROUP = MODE == MODE_FP8 ? 1 : BLOCK / EPV;        // lanes per FP4 block
    constexpr bool EXACT = MODE == MODE_FP8;
    // FP8 with W16: s * w is exact, so max |y| = RN(rstd * max |s w|) and the row max of |s w|
    // is reduced together with the sum of squares: one CTA barrier per row, y formed once in
    // the quantisation pass. Otherwise y is formed after rstd, kept in registers (up to four
    // vectors per thread) and its max reduced at a second barrier.
    constexpr bool ONE_BAR = MODE == MODE_FP8 && W16;
    // SCHED_WARP: every warp is its own row processor (rows, ring and mbarriers per warp); the
    // bulk-copy ring logic is shared with SCHED_PIPE.
    constexpr bool WARP_ROWS = SCHED == SCHED_WARP;
    constexpr bool CLUSTER = SCHED == SCHED_CLUSTER;
    constexpr bool RING = SCHED == SCHED_PIPE || WARP_ROWS || CLUSTER;
    // The ring schedules can keep the row in its shared-memory slot until the row is done: pass 1 writes
    // the residual sum s back over x and later passes re-read it, so no row data is held in
    // registers across the CTA barrier (the slot is refilled after an end-of-row barrier). That
    // pays except for the FP8 kernels with an offset or fp32 input (instruction-bound: they keep s
    // and y in registers and refill the slot right after the sum-of-squares barrier).
    //
    // The global-scale pre-pass needs no second pass over the row: each thread keeps
    // max |s w| of its elements from pass 1, and max |y| = RN(rstd * that) per thread (rstd > 0
    // and rounding is monotonic), so its slot is refilled right after the sum-of-squares
    // barrier. Its cluster schedule keeps the slot (PIPE_X finishes each row one row later).
    constexpr bool AMAX_P1 = MODE == MODE_AMAX && SCHED != SCHED_CLUSTER;
    constexpr bool SMEM_S = RING && (MODE != MODE_FP8 || W16) && !AMAX_P1;
    // NVFP4 with a ring: pass 2 is blocked, each thread owns whole 16-element scale blocks
    // (GROUP consecutive vectors, re-read from the slot), so the block scale, its table lookup
    // and its store happen once per block and the codes leave in one 8-byte store.
    constexpr bool NV_BLOCKED = MODE == MODE_NVFP4 && RING && VPT >= GROUP;
    constexpr bool KEEP_Y = VPT <= 4 && !ONE_BAR && !SMEM_S;
    // SCHED_CLUSTER with one exchange per row (every kernel that keeps s in its slot): the
    // exchange of a row overlaps the first pass of the next one (see the row loop).
    constexpr bool PIPE_X = CLUSTER && SMEM_S;
    // PIPE_X with a residual: the ring's slots hold x only (x becomes s and must live until its
    // row is finished, one row later), and the residual has a one-slot ring of its own, refilled
    // with the next row's residual as soon as the first pass is over. Two rows held plus one
    // loading then cost 3 x-slots + 1 residual slot instead of 3 slots of both.
    constexpr bool SPLIT_RES = PIPE_X && RES;

    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x;
    const int T = blockDim.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = T >> 5;
    const int rt = WARP_ROWS ? lane : tid;       // this thread's index within its row
    const int RT = WARP_ROWS ? 32 : T;           // threads per row
    // SCHED_CLUSTER: this CTA's slice of every row is vectors [voff, voff + nv) of stride
    const uint32_t crank = CLUSTER ? cluster_rank() : 0u;
    const uint32_t csize = CLUSTER ? cluster_size() : 1u;
    const int nv = CLUSTER ? p.nvec / static_cast<int>(csize) : p.nvec;   // vectors handled
    const long long stride = p.nvec;                                      // vectors per row
    const int voff = static_cast<int>(crank) * nv;
    const uint32_t row_bytes = static_cast<uint32_t>(nv) * 16u;
    const uint32_t stage_bytes = row_bytes * (RES && !SPLIT_RES ? 2u : 1u);
    const int S = RING ? p.stages : 0;
    const int nrings = WARP_ROWS ? nwarps : 1;
    // SPLIT_RES: the residual slot follows the ring; its mbarrier and row number are entry S of
    // the (then S + 1 long) barrier and row arrays
    const uint32_t rslot_bytes = SPLIT_RES ? row_bytes : 0u;
    const int SB = S + (SPLIT_RES ? 1 : 0);
    float* red = reinterpret_cast<float*>(smem + static_cast<size_t>(S) * nrings * stage_bytes + rslot_bytes);
    float2* red_ss_all = reinterpret_cast<float2*>(red);                    // [2][32]
    float* red_max_all = red + 128;                                         // [2][32]
    float* nv_factor = WARP_ROWS ? red : red + 192;                         // [128]

    uint64_t* bars_all =
        reinterpret_cast<uint64_t*>(red + (WARP_ROWS ? kRedFloatsWarp : kRedFloats));  // [nrings][S]
    long long* rows_all = reinterpret_cast<long long*>(bars_all + SB * nrings);       // [nrings][SB]
    // this thread's ring: its slots, its mbarriers, the row of each slot (-1: the ring is done),
    // the thread that refills it, and its rows
    unsigned char* ring = smem + (WARP_ROWS ? static_cast<size_t>(warp) * S * stage_bytes : 0);
    uint64_t* bars = bars_all + (WARP_ROWS ? warp * S : 0);
    long long* slot_rows = rows_all + (WARP_ROWS ? warp * S : 0);
    float4* xch = reinterpret_cast<float4*>(rows_all + SB * nrings);                 // [4]
    const uint32_t rslot = smem_u32(smem + static_cast<size_t>(S) * stage_bytes);   // SPLIT_RES
    const bool issuer = WARP_ROWS ? lane == 0 : tid == 0;
    const long long row0 = WARP_ROWS ? static_cast<long long>(blockIdx.x) * nwarps + warp
                           : CLUSTER ? static_cast<long long>(cluster_id())
                                     : static_cast<long long>(blockIdx.x);
    const long long rstep = WARP_ROWS ? static_cast<long long>(gridDim.x) * nwarps
                            : CLUSTER ? static_cast<long long>(cluster_count())
                                      : static_cast<long long>(gridDim.x);

    const uint4* __restrict__ xg = static_cast<const uint4*>(p.x) + voff;
    const uint4* __restrict__ rg = RES ? static_cast<const uint4*>(p.res) + voff : nullptr;
    uint4* __restrict__ rog = RES ? static_cast<uint4*>(p.res_out) + voff : nullptr;
    // first block scale of this CTA's slice (FP4), and the byte offset of its codes
    const int sf_off = voff * EPV / BLOCK;

    uint64_t policy = 0;
    if constexpr (RING) {
        policy = l2_evict_normal_policy();
        if (issuer) {
            for (int s = 0; s < SB; ++s) mbar_init(smem_u32(&bars[s]), 1);
            fence_mbar_init();
        }
    }
    // Programmatic dependent launch: everything above touches only shared memory and registers.
    // Wait here until the previous kernel on the stream has completed and its writes are
    // visible, then let the next one start its own prologue while this grid runs.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    // The ring's rows, as its refilling thread hands them out: round-robin over the row
    // processors below rows_static, then one at a time from the launch's counter; -1 when none
    // is left. Counter tickets are taken one call ahead, so the atomic's round trip overlaps a
    // whole row instead of delaying the refill. Each refilling thread stops at its first ticket
    // past the last row, so the counter sees exactly (rows - rows_static) + (row processors)
    // tickets; the thread holding the last of them is the last to touch it and sets it back to
    // 0 for the counter's next launch.
    long long next_static = row0;
    unsigned int ahead = 0;       // counter ticket taken for the next call
    bool have_ahead = false;
    bool exhausted = false;
    const unsigned long long last_ticket =
        static_cast<unsigned long long>(p.rows - p.rows_static) + static_cast<unsigned long long>(rstep) - 1;
    auto next_row = [&]() -> long long {
        if (exhausted) return -1;
        long long r;
        if (next_static < p.rows_static) {
            r = next_static;
            next_static += rstep;
            if (next_static >= p.rows_static && p.rowctr != nullptr) {
                ahead = atomicAdd(p.rowctr, 1u);
                have_ahead = true;
            }
        } else if (p.rowctr != nullptr) {
            const unsigned int t = have_ahead ? ahead : atomicAdd(p.rowctr, 1u);
            r = p.rows_static + static_cast<long long>(t);
            have_ahead = false;
            if (r >= p.rows) {
                exhausted = true;
                if (t == last_ticket) *p.rowctr = 0u;
                return -1;
            }
            ahead = atomicAdd(p.rowctr, 1u);
            have_ahead = true;
        } else {
            r = p.rows;
        }
        if (r >= p.rows) {
            exhausted = true;
            return -1;
        }
        return r;
    };
    // Give slot `st` (shared address `addr`) its next row: record the row number, then start the
    // copies, or complete the slot's phase empty-handed when the ring has no row left. `reuse`:
    // the slot's memory was read or written by threads before (order that before the copy).
    auto refill = [&](int st, uint32_t addr, bool reuse) {
        const long long r = next_row();
        slot_rows[st] = r;
        const uint32_t bar = smem_u32(&bars[st]);
        if (r < 0) {
            mbar_arrive(bar);
            return;
        }
        if (reuse) fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, stage_bytes);
        bulk_load(addr, xg + r * stride, row_bytes, bar, policy);
        if constexpr (RES && !SPLIT_RES) bulk_load(addr + row_bytes, rg + r * stride, row_bytes, bar, policy);
    };
    // SPLIT_RES: load row r's residual into the residual slot (r < 0: complete its phase empty).
    // Every acquisition of a ring slot pairs with one phase of the residual slot, in ring order.
    bool r_pending = false;       // (issuer) a residual phase not yet seen complete, and its parity
    uint32_t r_pend_par = 0;
    uint32_t rparity = 0;         // the residual slot's next phase parity (every thread)
    auto refill_res = [&](long long r, bool reuse) {
        const uint32_t bar = smem_u32(&bars[S]);
        slot_rows[S] = r;
        if (r < 0) {
            mbar_arrive(bar);
        } else {
            if (reuse) fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar, row_bytes);
            bulk_load(rslot, rg + r * stride, row_bytes, bar, policy);
        }
        r_pending = true;
        r_pend_par = rparity;
    };
    if constexpr (RING) {
        // the ring's first rows, issued by the thread that initialised its barriers
        if (issuer) {
            for (int s = 0; s < S; ++s)
                refill(s, smem_u32(ring + static_cast<size_t>(s) * stage_bytes), false);
            if constexpr (SPLIT_RES) refill_res(slot_rows[0], false);
        }
    }

    float gs = 1.0f, gs_over_6 = 0.0f;
    if constexpr (MODE == MODE_NVFP4) {
        gs = __ldg(p.gs);
        gs_over_6 = __fdiv_rn(gs, 6.0f);
        // factor[c] = gs / dec(c) for every positive E4M3 code (0 for code 0 and for NaN)
        for (int c = tid; c < 128; c += T) {
            const float ds = e4m3_value(static_cast<uint32_t>(c));
            nv_factor[c] = (c == 0 || c == 0x7F) ? 0.0f : __fdiv_rn(gs, ds);
        }
    }
    // the barrier initialisations and the factor table are visible to every thread after this
    if constexpr (RING || MODE == MODE_NVFP4) __syncthreads();

    const float2 offset2 = splat(p.offset);
    constexpr bool GAMMA_L1 = fp8_offset16<DT, MODE, VPT, SCHED, W16>();
    constexpr bool GAMMA_SMEM = GAMMA_L1 && SCHED == SCHED_PIPE;
    std::conditional_t<GAMMA_SMEM, GammaSmem<E, VPT>,
                       std::conditional_t<GAMMA_L1, GammaL1<E, VPT>, GammaRegs<E, VPT, !W16 && VPT <= 4>>> G;
    if constexpr (GAMMA_SMEM) {
        G.init(smem_u32(xch), static_cast<const uint4*>(p.gamma) + voff, rt, RT, nv, splat(p.offset));
        __syncthreads();
    }
    G.load(static_cast<const uint4*>(p.gamma) + voff, rt, RT, nv, offset2, NV_BLOCKED ? GROUP : 1);
    constexpr bool sw_exact = W16;                            // s * gamma exact in fp32
    const float Hf = static_cast<float>(p.hidden);
    // lanes in the second reduction stage: the smallest power of two >= nwarps
    int red_lanes = 1;
    while (red_lanes < nwarps) red_lanes <<= 1;

    // 1 / H: exact when H is a power of two (the FP8 exact path then skips the division)
    const bool h_pow2 = (p.hidden & (p.hidden - 1)) == 0;
    const float inv_h = __frcp_rn(Hf);

    float run_max = 0.0f;   // MODE_AMAX: max |y| over this thread's share of the CTA's rows
    int stage = 0;          // the next ring slot to wait on, and its mbarrier phase parity
    uint32_t parity = 0;
    int rbuf = 0;           // which of the two sum-of-squares reduction buffers this row uses
    bool aborted = false;   // a bounded wait ran out
    int cslot = 0;          // SCHED_CLUSTER: which of the three sum exchange slots this row posts to
    int mpar = 0;           // SCHED_CLUSTER: which of the two FP8 row amax slots this row uses
    // PIPE_X: the row whose exchange is in flight (-1: none), its ring slot, slot address and
    // exchange slot
    long long pend_row = -1;
    int pend_stage = 0;
    uint32_t pend_addr = 0;
    int pend_cslot = 0;
    long long reg_row = row0;
    for (;;) {
        // ---- which row: the slot's (ring schedules) or the next round-robin one --------------
        bool timed_out = false;
        uint32_t stage_addr = 0;
        const int cur_stage = stage;  // the slot acquired here (PIPE_X: the ring moves on at once)
        long long row;
        if constexpr (RING) {
            stage_addr = smem_u32(ring + static_cast<size_t>(stage) * stage_bytes);
            timed_out = !mbar_wait_bounded(smem_u32(&bars[stage]), parity, p.timeout_ns);
            if constexpr (SPLIT_RES) {
                // this acquisition's phase of the residual slot (empty when the slot is)
                const bool rok = mbar_wait_bounded(smem_u32(&bars[S]), rparity, p.timeout_ns);
                timed_out = timed_out || !rok;
                if (rok) r_pending = false;
                rparity ^= 1u;
            }
            // The slot's row number was written before its barrier was armed, and an empty slot
            // (-1) completes at once, so every thread of the ring reads the same value here.
            row = slot_rows[stage];
            if constexpr (PIPE_X) {
                if (++stage == S) {
                    stage = 0;
                    parity ^= 1u;
                }
            }
            // the ring handed out its last row (PIPE_X: once the row in flight is finished)
            if (row < 0 && (!PIPE_X || pend_row < 0)) break;
        } else {
            row = reg_row;
            reg_row += rstep;
            if (row >= p.rows) break;
        }
        // false after a timed-out wait (the loop then stops after the exchange that reports it)
        // and for the empty slot that ends a PIPE_X ring
        const bool have = PIPE_X ? !timed_out && row >= 0 : !timed_out;
        const uint4* __restrict__ xrow = xg + row * stride;
        const uint4* __restrict__ rrow = RES ? rg + row * stride : nullptr;
        // ---- load the row, add the residual, write residual_output, sum of squares ----------
        uint4 s[VPT];
        float2 acc_hi = make_float2(0.0f, 0.0f), acc_lo = make_float2(0.0f, 0.0f);
        float pmax = 0.0f;      // ONE_BAR and the pre-pass: max |s w| over this thread's elements
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = rt + k * RT;
            s[k] = make_uint4(0, 0, 0, 0);
            if (v < nv && have) {
                uint4 xv, rv;
                if constexpr (RING) {
                    xv = ld_shared_v4(stage_addr + v * 16u);
                    if constexpr (SPLIT_RES) rv = ld_shared_v4(rslot + v * 16u);
                    else if constexpr (RES) rv = ld_shared_v4(stage_addr + row_bytes + v * 16u);
                } else {
                    xv = ld_stream_v4(xrow + v);
                    if constexpr (RES) rv = ld_stream_v4(rrow + v);
                }
                if constexpr (RES) {
                    s[k] = E::add(xv, rv);
                    if constexpr (MODE != MODE_AMAX) st_v4(rog + row * stride + v, s[k]);
                    if constexpr (SMEM_S) st_shared_v4(stage_addr + v * 16u, s[k]);
                } else {
                    s[k] = xv;
                }
                if constexpr (W16) {
                    const uint32_t sv[4] = {s[k].x, s[k].y, s[k].z, s[k].w};
                    if constexpr (EXACT) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float2 sq = E::mul_halves(sv[j], sv[j]);   // exact squares
                            float2 t, e;
                            two_sum2(acc_hi, sq, t, e);
                            acc_hi = t;
                            acc_lo = add2(acc_lo, e);
                        }
                        if constexpr (ONE_BAR) {
                            const uint4 gk = G.packed(k);
                            const uint32_t gv[4] = {gk.x, gk.y, gk.z, gk.w};
                            float2 pw[NP];
#pragma unroll
                            for (int j = 0; j < NP; ++j) pw[j] = E::mul_halves(sv[j], gv[j]);
                            pmax = fmaxf(pmax, absmax_pairs(pw));
                        }
                    } else {
                        // two independent accumulator pairs shorten the dependency chain
                        acc_hi = E::sq_acc(sv[0], acc_hi);
                        acc_lo = E::sq_acc(sv[1], acc_lo);
                        acc_hi = E::sq_acc(sv[2], acc_hi);
                        acc_lo = E::sq_acc(sv[3], acc_lo);
                        if constexpr (AMAX_P1) {
                            const uint4 gk = G.packed(k);
                            const uint32_t gv[4] = {gk.x, gk.y, gk.z, gk.w};
                            float2 pw[NP];
#pragma unroll
                            for (int j = 0; j < NP; ++j) pw[j] = E::mul_halves(sv[j], gv[j]);
                            pmax = fmaxf(pmax, absmax_pairs(pw));
                        }
                    }
                } else if constexpr (EXACT && DT != DT_F32) {
                    // exact squares straight from the packed halves (mixed-precision FMA)
                    const uint32_t sv[4] = {s[k].x, s[k].y, s[k].z, s[k].w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float2 sq = E::mul_halves(sv[j], sv[j]);
                        float2 t, e;
                        two_sum2(acc_hi, sq, t, e);
                        acc_hi = t;
                        acc_lo = add2(acc_lo, e);
                    }
                } else {
                    float2 f[NP];
                    E::pairs(s[k], f);
#pragma unroll
                    for (int j = 0; j < NP; ++j) {
                        if constexpr (EXACT) {
                            const float2 sq = mul2(f[j], f[j]);          // fp32: hi part of f^2
                            float2 t, e;
                            two_sum2(acc_hi, sq, t, e);
                            acc_hi = t;
                            acc_lo = add2(acc_lo, e);
                            if constexpr (DT == DT_F32)
                                acc_lo = add2(acc_lo, fma2(f[j], f[j], make_float2(-sq.x, -sq.y)));
                        } else {
                            acc_hi = fma2(f[j], f[j], acc_hi);
                        }
                    }
                    if constexpr (AMAX_P1) {
                        float2 w[NP];
                        G.get(k, w);
#pragma unroll
                        for (int j = 0; j < NP; ++j) f[j] = mul2(f[j], w[j]);
                        pmax = fmaxf(pmax, absmax_pairs(f));
                    }
                }
            }
        }
        // ---- CTA reduction of the sum of squares -> rstd ----------------------------------
        float2* red_ss = red_ss_all + rbuf * 32;
        float* red_max = red_max_all + rbuf * 32;
        rbuf ^= 1;
        if constexpr (ONE_BAR) {
            pmax = warp_max_abs(pmax);
            if (!WARP_ROWS && lane == 0) red_max[warp] = pmax;
        }
        FF ss;
        if constexpr (EXACT) {
            ss = ff_add(FF{acc_hi.x, acc_lo.x}, FF{acc_hi.y, acc_lo.y});
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss = ff_add_pos(ss, shfl_xor_ff(ss, o));
        } else {
            ss = FF{warp_sum(__fadd_rn(__fadd_rn(acc_hi.x, acc_hi.y), __fadd_rn(acc_lo.x, acc_lo.y))), 0.0f};
        }
        if (!WARP_ROWS && lane == 0) red_ss[warp] = make_float2(ss.hi, ss.lo);
        bool stop;
        // the row's FP8 scale from its amax (rounded to the scale output type, whose value the
        // codes are formed against), stored by `writer`
        auto fp8_scale = [&](float amax, bool writer) -> float {
            float sc = __fdiv_rn(fminf(amax, p.scale_ub), 448.0f);
            if (p.scale_dtype == DT_BF16) {
                uint16_t h;
                asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(sc));
                sc = __uint_as_float(static_cast<uint32_t>(h) << 16);
                if (writer) static_cast<uint16_t*>(p.scale_out)[row] = h;
            } else if (p.scale_dtype == DT_FP16) {
                uint16_t h;
                asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(sc));
                asm("cvt.f32.f16 %0, %1;" : "=f"(sc) : "h"(h));
                if (writer) static_cast<uint16_t*>(p.scale_out)[row] = h;
            } else {
                if (writer) static_cast<float*>(p.scale_out)[row] = sc;
            }
            return sc;
        };
        if constexpr (WARP_ROWS) stop = __any_sync(0xFFFFFFFFu, timed_out);
        else stop = __syncthreads_or(timed_out);
        if constexpr (SPLIT_RES) {
            // every thread is past its reads of the residual slot: load the next acquisition's
            // residual now (not after a timed-out wait: the CTA stops below)
            if (issuer && !stop) refill_res(slot_rows[stage], true);
        }
        // the row's (or, for SCHED_CLUSTER, this CTA's slice's) sum of squares and ONE_BAR max,
        // the same in every thread
        FF tot = ss;
        float tmax = pmax;
        if constexpr (!WARP_ROWS) {
            const float2 part = lane < nwarps ? red_ss[lane] : make_float2(0.0f, 0.0f);
            if constexpr (EXACT) {
                FF t{part.x, part.y};
#pragma unroll
                for (int o = 8; o > 0; o >>= 1)
                    if (o < red_lanes) t = ff_add_pos(t, shfl_xor_ff(t, o));
                tot.hi = __shfl_sync(0xFFFFFFFFu, t.hi, 0);
                tot.lo = __shfl_sync(0xFFFFFFFFu, t.lo, 0);
                if constexpr (ONE_BAR) {
                    float m = lane < nwarps ? red_max[lane] : 0.0f;
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1)
                        if (o < red_lanes) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
                    tmax = __shfl_sync(0xFFFFFFFFu, m, 0);
                }
            } else {
                float t = part.x;
#pragma unroll
                for (int o = 8; o > 0; o >>= 1)
                    if (o < red_lanes) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
                tot = FF{__shfl_sync(0xFFFFFFFFu, t, 0), 0.0f};
            }
        }
        // the row finished below and its ring slot: this row, or (PIPE_X) the one posted last time
        int fin_stage = PIPE_X ? cur_stage : stage;
        if constexpr (CLUSTER) {
            // The cluster's CTAs trade their slice totals (and whether any wait ran out): each
            // writes its own slot, passes the cluster barrier, then every CTA adds the C slots in
            // rank order, so all of them hold the same row totals and take the same branch below.
            float4* slot = &xch[cslot];
            const int my_cslot = cslot;
            if (++cslot == 3) cslot = 0;
            auto gather = [&](const float4* sl) {
                FF sum{0.0f, 0.0f};
                float mx = 0.0f;
                bool any = false;
                for (uint32_t k = 0; k < csize; ++k) {
                    const float4 v = ld_cluster_f4(smem_u32(sl), k);
                    if constexpr (EXACT) sum = ff_add(sum, FF{v.x, v.y});
                    else sum.hi = __fadd_rn(sum.hi, v.x);
                    mx = fmaxf(mx, v.z);
                    any = any || v.w != 0.0f;
                }
                tot = sum;
                tmax = mx;
                stop = any;
            };
            if constexpr (PIPE_X) {
                // Row i posts its totals, waits for the exchange of row i - 1 (posted one
                // iteration ago, so its barrier had this row's first pass to complete), arrives
                // for row i, then finishes row i - 1. Every CTA of the cluster walks the same rows
                // and so makes the same barrier calls: arrive(0), wait(0) arrive(1), ...,
                // wait(n - 1), then the final barrier. A slot is rewritten three rows later, after
                // a barrier that every CTA passed only once done reading it.
                // Only thread 0 writes what other CTAs read (the slot), so only it arrives with
                // release semantics. The others arrive relaxed: their loads of the previous slots
                // decide whether they arrive at all, so those loads are complete by then.
                const bool publish = tid == 0;
                const bool post = row >= 0;
                if (post && tid == 0) *slot = make_float4(tot.hi, tot.lo, tmax, stop ? 1.0f : 0.0f);
                if (pend_row < 0) {
                    // the first row: nothing to finish yet
                    cluster_arrive_as(publish);
                    pend_row = row;
                    pend_stage = cur_stage;
                    pend_addr = stage_addr;
                    pend_cslot = my_cslot;
                    continue;
                }
                cluster_wait();
                gather(&xch[pend_cslot]);
                if (post && !stop) cluster_arrive_as(publish);
                fin_stage = pend_stage;
                const long long next_row_id = row;
                const uint32_t next_addr = stage_addr;
                row = pend_row;
                stage_addr = pend_addr;
                pend_row = next_row_id;
                pend_stage = cur_stage;
                pend_addr = next_addr;
                pend_cslot = my_cslot;
            } else {
                // As above, only the slot writer arrives with release semantics; the others'
                // reads of earlier slots were consumed (the stop decision, the row's scale)
                // before they arrive again.
                if (tid == 0) *slot = make_float4(tot.hi, tot.lo, tmax, stop ? 1.0f : 0.0f);
                cluster_arrive_as(tid == 0);
                cluster_wait();
                gather(slot);
            }
        }
        if (stop) {
            if constexpr (RING) {
                if (issuer) {
                    atomicOr(p.err, ERRF_WAIT_TIMEOUT);
                    // Before the CTA exits, let every copy it issued land: the slot whose wait ran
                    // out and every later one (PIPE_X: from the slot acquired last, the ring
                    // having moved past it). Each slot has one phase outstanding; a slot that is
                    // already complete, or was armed empty, passes at once. These waits take four
                    // times the bound; one that runs out as well is recorded, because the CTA
                    // then exits with a copy into its shared memory possibly still pending.
                    int js = stage;
                    uint32_t jp = parity;
                    int n = S;
                    if constexpr (PIPE_X) {
                        // back to the slot acquired last (cur_stage), then the S - 2 after it
                        if (js == 0) {
                            js = S - 1;
                            jp ^= 1u;
                        } else {
                            --js;
                        }
                        n = S - 1;
                    }
                    bool drained = true;
                    if constexpr (SPLIT_RES) {
                        if (r_pending)
                            drained = mbar_wait_bounded(smem_u32(&bars[S]), r_pend_par, 4 * p.timeout_ns);
                    }
                    for (int j = 0; j < n; ++j) {
                        drained = mbar_wait_bounded(smem_u32(&bars[js]), jp, 4 * p.timeout_ns) && drained;
                        if (++js == S) {
                            js = 0;
                            jp ^= 1u;
                        }
                    }
                    if (!drained) atomicOr(p.err, ERRF_DRAIN_TIMEOUT);
                }
            }
            aborted = true;
            break;
        }
        if constexpr (RING && !SMEM_S) {
            // Every thread has read this slot (s is held in registers): refill it now.
            if constexpr (WARP_ROWS) __syncwarp();
            if (issuer) refill(fin_stage, stage_addr, true);
        }
        float rstd;
        if constexpr (EXACT)
            rstd = h_pow2 ? rstd_from_sum_pow2(tot, inv_h, p.eps) : rstd_from_sum(tot, Hf, p.eps);
        else
            rstd = __frsqrt_rn(__fadd_rn(__fmul_rn(tot.hi, inv_h), p.eps));
        if constexpr (ONE_BAR) pmax = tmax;
        const float2 rstd2 = splat(rstd);
        // the residual sum s of vector k (zero past the row end)
        auto get_s = [&](int k) -> uint4 {
            if constexpr (SMEM_S) {
                const int v = rt + k * RT;
                return v < nv ? ld_shared_v4(stage_addr + v * 16u) : make_uint4(0, 0, 0, 0);
            } else {
                return s[k];
            }
        };
        // s * w for the pairs of vector k (exact when W16)
        auto sw_pairs = [&](int k, float2 (&out)[NP]) {
            const uint4 sk = get_s(k);
            if constexpr (W16) {
                const uint32_t sv[4] = {sk.x, sk.y, sk.z, sk.w};
                const uint4 gk = G.packed(k);
                            const uint32_t gv[4] = {gk.x, gk.y, gk.z, gk.w};
#pragma unroll
                for (int j = 0; j < NP; ++j) out[j] = E::mul_halves(sv[j], gv[j]);
            } else {
                float2 f[NP], w[NP];
                E::pairs(sk, f);
                G.get(k, w);
#pragma unroll
                for (int j = 0; j < NP; ++j) out[j] = mul2(f[j], w[j]);
            }
        };

        if constexpr (MODE == MODE_AMAX) {
            // max |y| = rstd * max |s w| (rstd > 0, rounding is monotonic)
            float mp = pmax;
            if constexpr (!AMAX_P1) {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    float2 sw[NP];
                    sw_pairs(k, sw);
                    mp = fmaxf(mp, absmax_pairs(sw));
                }
            }
            if (mp > 0.0f) run_max = fmaxf(run_max, __fmul_rn(mp, rstd));
        } else if constexpr (MODE == MODE_FP8) {
            // ---- y, row amax, scale, E4M3 codes ----------------------------------------------
            // With 16-bit inputs and weight_offset 0, s * w is exact and y = RN(RN(s w) rstd) is
            // already the correctly rounded product; otherwise the FMA split forms it.
            float2 y[KEEP_Y ? VPT : 1][NP];
            float amax = 0.0f;
            if constexpr (ONE_BAR) {
                amax = pmax > 0.0f ? __fmul_rn(pmax, rstd) : 0.0f;   // = max |RN(s w rstd)|
            } else {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    float2 yy[NP];
                    if constexpr (sw_exact) {
                        sw_pairs(k, yy);
#pragma unroll
                        for (int j = 0; j < NP; ++j) yy[j] = mul2(yy[j], rstd2);
                    } else {
                        float2 f[NP], w[NP];
                        E::pairs(get_s(k), f);
                        G.get(k, w);
#pragma unroll
                        for (int j = 0; j < NP; ++j) yy[j] = norm_mul2(f[j], w[j], rstd2);
                    }
                    if constexpr (KEEP_Y) {
#pragma unroll
                        for (int j = 0; j < NP; ++j) y[k][j] = yy[j];
                    }
                    amax = fmaxf(amax, absmax_pairs(yy));
                }
                amax = warp_max_abs(amax);
                if constexpr (!WARP_ROWS) {
                    if (lane == 0) red_max[warp] = amax;
                    __syncthreads();
                    amax = lane < nwarps ? red_max[lane] : 0.0f;
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1)
                        if (o < red_lanes) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
                    amax = __shfl_sync(0xFFFFFFFFu, amax, 0);
                }
                if constexpr (CLUSTER) {
                    float4* slot = &xch[3 + mpar];
                    mpar ^= 1;
                    if (tid == 0) *slot = make_float4(amax, 0.0f, 0.0f, 0.0f);
                    cluster_arrive_as(tid == 0);
                    cluster_wait();
                    float mx = 0.0f;
                    for (uint32_t k = 0; k < csize; ++k) mx = fmaxf(mx, ld_cluster_f4(smem_u32(slot), k).x);
                    amax = mx;
                }
            }
            const float scale = fp8_scale(amax, rt == 0 && crank == 0);
            const float inv = scale > 0.0f ? __frcp_rn(scale) : 0.0f;
            // a zero scale (all-zero row) gives inv = 0, so every quotient below is a zero and
            // every code 0x00 (or 0x80 for a negative zero y: the same value)
            const float2 inv2 = splat(inv);
            const float2 nd2 = splat(-scale);
            unsigned char* outp = static_cast<unsigned char*>(p.out) + row * p.hidden +
                                  static_cast<long long>(voff) * EPV;
            // y of vector k of this thread
            auto y_of = [&](int k, float2 (&yk)[NP]) {
                if constexpr (KEEP_Y) {
#pragma unroll
                    for (int j = 0; j < NP; ++j) yk[j] = y[k][j];
                } else if constexpr (sw_exact) {
                    sw_pairs(k, yk);
#pragma unroll
                    for (int j = 0; j < NP; ++j) yk[j] = mul2(yk[j], rstd2);
                } else {
                    float2 f[NP], w[NP];
                    E::pairs(get_s(k), f);
                    G.get(k, w);
#pragma unroll
                    for (int j = 0; j < NP; ++j) yk[j] = norm_mul2(f[j], w[j], rstd2);
                }
            };
            auto store_codes = [&](int v, const float2 (&q)[NP]) {
                uint32_t c[NP];
#pragma unroll
                for (int j = 0; j < NP; ++j) c[j] = cvt_e4m3x2(q[j].x, q[j].y);
                if constexpr (EPV == 8) {
                    st_v2(outp + v * 8, c[0] | (c[1] << 16), c[2] | (c[3] << 16));
                } else {
                    st_u32(outp + v * 4, c[0] | (c[1] << 16));
                }
            };
            if constexpr (W16) {
                // With 16-bit products, quotients land exactly on an E4M3 boundary often enough
                // (448 * P_i / P_max, a ratio of short numbers) that the fix-up stays per vector,
                // on the 8 values at hand.
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int v = rt + k * RT;
                    if (v >= nv) continue;
                    float2 yk[NP], q[NP];
                    y_of(k, yk);
                    uint32_t key = 0xFFFFFFFFu;
#pragma unroll
                    for (int j = 0; j < NP; ++j) {
                        q[j] = div_rn2(yk[j], nd2, inv2);
                        key = min(key, min(tie_key(q[j].x), tie_key(q[j].y)));
                    }
                    if (key == 0u) {
#pragma unroll
                        for (int j = 0; j < NP; ++j) {
                            q[j].x = untie(q[j].x, yk[j].x, nd2.x);
                            q[j].y = untie(q[j].y, yk[j].y, nd2.y);
                        }
                    }
                    store_codes(v, q);
                }
            } else {
                // Otherwise such quotients are rare (about 2^-19 of them), so the common path has
                // no branch per vector and the vectors' work interleaves: the correctly rounded
                // quotients go straight to E4M3 and the tie keys are folded over the row. A
                // thread that met a boundary redoes its vectors with the fix-up and stores them
                // again.
                uint32_t key = 0xFFFFFFFFu;
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int v = rt + k * RT;
                    if (v >= nv) continue;
                    float2 yk[NP], q[NP];
                    y_of(k, yk);
#pragma unroll
                    for (int j = 0; j < NP; ++j) {
                        q[j] = div_rn2(yk[j], nd2, inv2);
                        key = min(key, min(tie_key(q[j].x), tie_key(q[j].y)));
                    }
                    store_codes(v, q);
                }
                if (key == 0u) {
#pragma unroll
                    for (int k = 0; k < VPT; ++k) {
                        const int v = rt + k * RT;
                        if (v >= nv) continue;
                        float2 yk[NP], q[NP];
                        y_of(k, yk);
#pragma unroll
                        for (int j = 0; j < NP; ++j) {
                            q[j] = div_rn2(yk[j], nd2, inv2);
                            q[j].x = untie(q[j].x, yk[j].x, nd2.x);
                            q[j].y = untie(q[j].y, yk[j].y, nd2.y);
                        }
                        store_codes(v, q);
                    }
                }
            }
        } else if constexpr (NV_BLOCKED) {
            // ---- NVFP4, blocked: thread owns blocks b = rt + kb * RT (GROUP vectors each) -------
            unsigned char* outp = static_cast<unsigned char*>(p.out) + row * (p.hidden / 2) +
                                  static_cast<long long>(voff) * EPV / 2;
            unsigned char* sp_row = static_cast<unsigned char*>(p.scale_out) +
                (p.swizzled ? (row >> 7) * (static_cast<long long>(p.k_tiles) * 512) +
                                  (row & 31) * 16 + ((row & 127) >> 5) * 4
                            : row * p.nsf);
            const int nb = nv / GROUP;
#pragma unroll
            for (int kb = 0; kb < VPT / GROUP; ++kb) {
                const int b = rt + kb * RT;
                if (b >= nb) continue;
                float2 sw[GROUP][NP];
                float m = 0.0f;
#pragma unroll
                for (int j = 0; j < GROUP; ++j) {
                    const uint4 sk = ld_shared_v4(stage_addr + (b * GROUP + j) * 16u);
                    const int k = kb * GROUP + j;
                    if constexpr (W16) {
                        const uint32_t sv[4] = {sk.x, sk.y, sk.z, sk.w};
                        const uint4 gk = G.packed(k);
                            const uint32_t gv[4] = {gk.x, gk.y, gk.z, gk.w};
#pragma unroll
                        for (int i = 0; i < NP; ++i) sw[j][i] = E::mul_halves(sv[i], gv[i]);
                    } else {
                        float2 f[NP], w[NP];
                        E::pairs(sk, f);
                        G.get(k, w);
#pragma unroll
                        for (int i = 0; i < NP; ++i) sw[j][i] = mul2(f[i], w[i]);
                    }
                    m = fmaxf(m, absmax_pairs(sw[j]));
                }
                const float a = m > 0.0f ? __fmul_rn(m, rstd) : 0.0f;      // block max |y|
                const float t = fminf(__fmul_rn(a, gs_over_6), 448.0f);
                const uint32_t code = cvt_e4m3x2(t, 0.0f) & 0xFFu;
                const float factor = nv_factor[code & 0x7Fu];
                const int gb = sf_off + b;                                 // block in the row
                sp_row[p.swizzled ? (gb >> 2) * 512 + (gb & 3) : gb] = static_cast<unsigned char>(code);
                const bool zero_block = !(factor > 0.0f);
                const float2 f2 = splat(zero_block ? 0.0f : __fmul_rn(factor, rstd));
                uint32_t packed[GROUP];
#pragma unroll
                for (int j = 0; j < GROUP; ++j) {
                    if constexpr (EPV == 8) {
                        float q[8];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float2 qq = mul2(sw[j][i], f2);
                            q[2 * i] = qq.x;
                            q[2 * i + 1] = qq.y;
                        }
                        packed[j] = zero_block ? 0u : cvt_e2m1x8(q);
                    } else {
                        float q[4];
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            const float2 qq = mul2(sw[j][i], f2);
                            q[2 * i] = qq.x;
                            q[2 * i + 1] = qq.y;
                        }
                        packed[j] = zero_block ? 0u : cvt_e2m1x4(q);
                    }
                }
                if constexpr (EPV == 8) {
                    st_v2(outp + b * 8, packed[0], packed[1]);
                } else {
                    st_v2(outp + b * 8, packed[0] | (packed[1] << 16), packed[2] | (packed[3] << 16));
                }
            }
        } else {
            // ---- FP4: per-block amax across GROUP adjacent lanes, scale, E2M1 ---------------
            // The block max of y is rstd * max |s w|, and the codes are E2M1(s w * rstd * factor)
            // with rstd folded into the block factor: for MXFP4 the factor is a power of two, so
            // the codes equal E2M1(RN(s w rstd) * 2^(127 - e)) whenever s w is exact.
            unsigned char* outp = static_cast<unsigned char*>(p.out) + row * (p.hidden / 2) +
                                  static_cast<long long>(voff) * EPV / 2;
            // scale byte of block sf sits at sp_row + col(sf): row-major sp + row * nsf + sf, or
            // the swizzled 128x4 tile position (row part here, scale part per block)
            unsigned char* sp_row = static_cast<unsigned char*>(p.scale_out) +
                (p.swizzled ? (row >> 7) * (static_cast<long long>(p.k_tiles) * 512) +
                                  (row & 31) * 16 + ((row & 127) >> 5) * 4
                            : row * p.nsf);
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = rt + k * RT;
                float2 sw[NP];
                float m = 0.0f;
                sw_pairs(k, sw);
                m = absmax_pairs(sw);
#pragma unroll
                for (int o = 1; o < GROUP; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
                const float a = m > 0.0f ? __fmul_rn(m, rstd) : 0.0f;      // block max |y|
                float factor;
                uint32_t code;
                if constexpr (MODE == MODE_NVFP4) {
                    const float t = fminf(__fmul_rn(a, gs_over_6), 448.0f);
                    code = cvt_e4m3x2(t, 0.0f) & 0xFFu;
                    factor = nv_factor[code & 0x7Fu];
                } else {
                    code = ue8m0_code(a);
                    factor = ue8m0_inv_factor(code);
                }
                if (v >= nv) continue;
                if ((v & (GROUP - 1)) == 0)
                {
                    const int sf = sf_off + v / GROUP;
                    sp_row[p.swizzled ? (sf >> 2) * 512 + (sf & 3) : sf] = static_cast<unsigned char>(code);
                }
                const bool zero_block = !(factor > 0.0f);
                const float2 f2 = splat(zero_block ? 0.0f : __fmul_rn(factor, rstd));
                if constexpr (EPV == 8) {
                    float q[8];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float2 qq = mul2(sw[j], f2);
                        q[2 * j] = qq.x;
                        q[2 * j + 1] = qq.y;
                    }
                    st_u32(outp + v * 4, zero_block ? 0u : cvt_e2m1x8(q));
                } else {
                    float q[4];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float2 qq = mul2(sw[j], f2);
                        q[2 * j] = qq.x;
                        q[2 * j + 1] = qq.y;
                    }
                    st_u16(outp + v * 2, static_cast<uint16_t>(zero_block ? 0u : cvt_e2m1x4(q)));
                }
            }
        }
        if constexpr (SMEM_S) {
            // Every thread is done with this slot: refill it with the ring's next row.
            // (Each lane wrote s into the slot; in the row-per-warp schedule every lane orders
            // its writes before the refill's async-proxy writes.)
            if constexpr (WARP_ROWS) {
                fence_proxy_async_smem();
                __syncwarp();
            } else {
                __syncthreads();
            }
            if (issuer) refill(fin_stage, stage_addr, true);
        }
        if constexpr (PIPE_X) {
            if (pend_row < 0) break;      // the row just finished was the last
        } else if constexpr (RING) {
            if (++stage == S) {
                stage = 0;
                parity ^= 1u;
            }
        }
    }
    if constexpr (CLUSTER) cluster_sync();   // no CTA leaves while others may read its slots
    if constexpr (MODE == MODE_AMAX) {
        // The CTA's max |y| joins the launch's running max (non-negative floats order like their
        // bit patterns, so an unsigned max is a float max); then the CTA counts itself done. The
        // last CTA to do so reads the max, writes gs = 448 * 6 / max (1 for an all-zero tensor)
        // and leaves both words at 0 for the slot's next launch. A CTA stopped by a timed-out
        // wait still counts itself (the error word already reports the launch).
        const float wm = warp_max_abs(run_max);
        __syncthreads();                       // every warp is out of the row loop: `red` is free
        if (lane == 0) red[warp] = wm;
        __syncthreads();
        if (tid == 0) {
            float cm = 0.0f;
            for (int w = 0; w < nwarps; ++w) cm = fmaxf(cm, red[w]);
            if (!aborted && cm > 0.0f) atomicMax(p.amax_slot, __float_as_uint(cm));
            __threadfence();
            const unsigned int done = atomicAdd(p.amax_slot + 1, 1u);
            if (done == gridDim.x - 1) {
                __threadfence();
                const float amax = __uint_as_float(atomicExch(p.amax_slot, 0u));
                atomicExch(p.amax_slot + 1, 0u);
                *static_cast<float*>(p.scale_out) = amax > 0.0f ? __fdiv_rn(448.0f * 6.0f, amax) : 1.0f;
            }
        }
        return;
    }
    if (aborted) return;
}

}  // namespace rmsq
