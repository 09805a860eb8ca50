// rmsq_api.cu -- the C ABI of librmsq.so: argument checks, launch planning, the entry points
// declared in include/rmsq.h, and a few small diagnostic kernels.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "rmsq.h"
#include "rmsq_host.h"

namespace rmsq {

// Device-side error word (bit ERRF_WAIT_TIMEOUT: a bounded wait ran out). One per device.
static __device__ unsigned int g_err_word;

// Row counters of the dynamic row tail, one per launch, taken in turn from a pool of
// kCounterSlots slots (32 bytes apart) that lives as long as the library. The thread holding a
// launch's last ticket sets its counter back to 0, so a slot is clean when its turn comes again:
// launches in one stream run in order, and launches on other streams would have to be more than
// kCounterSlots launches apart in issue order and still running together to meet on a slot. A
// launch stopped by a timed-out wait can leave its counter behind; rmsq_device_status clears the
// pool when it reports that.
constexpr int kCounterSlots = 4096;
static __device__ __align__(256) unsigned int g_row_counters[kCounterSlots * 8];
static std::atomic<unsigned long long> g_counter_seq{0};

static std::atomic<int> g_schedule{0};
static std::atomic<int> g_tune_stages{0};
static std::atomic<int> g_tune_ctas{0};
static std::atomic<int> g_tune_vpt{0};
static std::atomic<int> g_tune_warps{0};
static std::atomic<int> g_tune_cluster{0};
static std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
static std::atomic<unsigned long long> g_launches{0};
static std::atomic<bool> g_pdl{true};
static std::atomic<bool> g_dynamic_rows{true};

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    bool usable = false;
    int sms = 0;
    int smem_optin = 0;
    int smem_per_sm = 0;       // shared memory of one SM
    int smem_reserved = 0;     // shared memory the system reserves per CTA
    unsigned int* err = nullptr;
    unsigned int* counters = nullptr;
};

static std::mutex g_mu;
static DeviceInfo g_dev[kMaxDevices];

// Per-device facts, read once with the device current: SM count, opt-in shared memory, the
// address of this device's error word, and whether the device is compute capability 10.3.
static const DeviceInfo* device_info()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        bool ok = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) ==
                      cudaSuccess &&
                  cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) ==
                      cudaSuccess &&
                  cudaDeviceGetAttribute(&d.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) ==
                      cudaSuccess;
        void* addr = nullptr;
        void* ctr = nullptr;
        ok = ok && major == 10 && minor == 3 &&
             cudaGetSymbolAddress(&addr, g_err_word) == cudaSuccess &&
             cudaGetSymbolAddress(&ctr, g_row_counters) == cudaSuccess;
        d.err = static_cast<unsigned int*>(addr);
        d.counters = static_cast<unsigned int*>(ctr);
        d.usable = ok;
        d.ready = true;
        if (!ok) cudaGetLastError();
    }
    return d.usable ? &d : nullptr;
}

struct OccEntry {
    const void* fn;
    int dev, threads, smem, cluster, blocks;   // blocks: per SM, or active clusters (cluster > 1)
    bool attr_set;
};
static OccEntry g_occ[512];
static int g_nocc = 0;

cudaError_t run_kernel(const void* fn, const Plan& pl, const Params& p, cudaStream_t stream)
{
    int dev = 0;
    cudaGetDevice(&dev);
    const DeviceInfo& di = g_dev[dev];
    int blocks = 0;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        int i = 0;
        const int cl = pl.sched == SCHED_CLUSTER ? pl.cluster : 1;
        for (; i < g_nocc; ++i)
            if (g_occ[i].fn == fn && g_occ[i].dev == dev && g_occ[i].threads == pl.threads &&
                g_occ[i].smem == pl.smem && g_occ[i].cluster == cl)
                break;
        if (i == g_nocc) {
            cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 di.smem_optin);
            if (e != cudaSuccess) return e;
            // The kernels stage rows in shared memory and barely use L1: prefer the largest
            // shared-memory carveout so the row rings of several CTAs fit on one SM.
            e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
            if (e != cudaSuccess) return e;
            if (cl > 8) {
                // clusters of 16 CTAs are beyond the portable size of 8
                e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                if (e != cudaSuccess) return e;
            }
            int b = 0;
            if (cl > 1) {
                // how many clusters of cl CTAs can be resident at once
                cudaLaunchConfig_t oc = {};
                oc.gridDim = dim3(static_cast<unsigned>(cl));
                oc.blockDim = dim3(pl.threads);
                oc.dynamicSmemBytes = static_cast<size_t>(pl.smem);
                cudaLaunchAttribute ca[1];
                ca[0].id = cudaLaunchAttributeClusterDimension;
                ca[0].val.clusterDim.x = static_cast<unsigned>(cl);
                ca[0].val.clusterDim.y = 1;
                ca[0].val.clusterDim.z = 1;
                oc.attrs = ca;
                oc.numAttrs = 1;
                e = cudaOccupancyMaxActiveClusters(&b, fn, &oc);
            } else {
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, pl.threads, pl.smem);
            }
            if (e != cudaSuccess) return e;
            if (g_nocc < static_cast<int>(sizeof(g_occ) / sizeof(g_occ[0])))
                g_occ[g_nocc++] = OccEntry{fn, dev, pl.threads, pl.smem, cl, b, true};
            blocks = b;
        } else {
            blocks = g_occ[i].blocks;
        }
    }
    if (blocks < 1) return cudaErrorInvalidConfiguration;
    long long grid;
    if (pl.sched == SCHED_CLUSTER) {
        // one cluster per row at a time; as many clusters as can be resident, at most one per row
        const long long clusters = p.rows < blocks ? p.rows : blocks;
        grid = clusters * pl.cluster;
    } else {
        if (pl.ctas_per_sm > 0 && blocks > pl.ctas_per_sm) blocks = pl.ctas_per_sm;
        grid = static_cast<long long>(blocks) * di.sms;
    }
    const long long rows_per_cta = pl.sched == SCHED_WARP ? pl.threads / 32 : 1;
    if (pl.sched != SCHED_CLUSTER && grid > (p.rows + rows_per_cta - 1) / rows_per_cta)
        grid = (p.rows + rows_per_cta - 1) / rows_per_cta;
    // Dynamic row tail (CTA-per-row ring schedule): SMs do not get equal shares of HBM
    // bandwidth, so with rows dealt out round-robin the slowest SM sets the end of the launch
    // (measured on GB300: the last CTA ended 11-17 us after the median one on 130-170 us
    // launches). Each CTA takes its first 3/4 of an equal share round-robin and the rest one
    // row at a time from the launch's counter.
    Params q = p;
    const long long procs = grid * rows_per_cta;
    q.rowctr = nullptr;
    q.rows_static = p.rows;
    // this launch's scratch slot of the pool: [0] the row counter, [1..2] the pre-pass's max
    // and done count
    unsigned int* slot = nullptr;
    if (di.counters != nullptr)
        slot = di.counters + (g_counter_seq.fetch_add(1) % kCounterSlots) * 8;
    q.amax_slot = slot != nullptr ? slot + 1 : nullptr;
    if (g_dynamic_rows.load() && pl.sched == SCHED_PIPE && slot != nullptr && p.rows >= 2 * procs &&
        p.rows < (1LL << 31)) {
        // a counter the caller set up (zeroed, on this stream) is used as it is
        q.rowctr = p.rowctr != nullptr ? p.rowctr : slot;
        q.rows_static = p.rows / procs * 3 / 4 * procs;
    }
    void* args[] = {&q};
    // Programmatic dependent launch: the kernel may be scheduled while the previous kernel on the
    // stream finishes; it waits (griddepcontrol.wait) before touching global memory.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(pl.threads);
    cfg.dynamicSmemBytes = static_cast<size_t>(pl.smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = g_pdl.load() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (pl.sched == SCHED_CLUSTER) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(pl.cluster);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
    return e;
}

// ------------------------------------------------------------------------------------------
// Planning
// ------------------------------------------------------------------------------------------

static int elems_per_vec(int dt) { return dt == DT_F32 ? 4 : 8; }

// Pick vectors per thread, CTA size, schedule, ring depth and residency for one call.
// From on-GPU sweeps (GB300), with nv = 16-byte vectors per row:
//  - Short rows (nv <= 256 without a residual, nv <= 64 with one) take the row-per-warp
//    schedule: 8 warps per CTA, a two-row ring per warp, as many CTAs as fit.
//  - Otherwise a CTA per row. Each thread takes the power of two nearest nv / 128 vectors
//    (FP8 without W16 at most 4, so y stays in registers), with two exceptions:
//    - FP4 with a residual: 2 vectors per thread up to 1024 vectors per row, then as many as
//      make 512 threads (NVFP4 rows of up to 512 vectors: 4; MXFP4 rows of up to 256: 1);
//    - FP8 rows of up to 256 vectors: 4 vectors per thread and about 12 warps per SM.
//  - A two-row ring per CTA; three for FP4 rows with a residual of 2048 vectors and more (one
//    CTA per SM then); the FP8 kernel with a weight offset and 16-bit input: one or two slots
//    beside its w table (below).
//  - CTAs per SM (shared memory permitting):
//    - FP4 with a residual: 8;
//    - the W16 FP8 kernel: 8 (measured on GB300 at 8192 x 4096: 37.5 us against 41.6 us with
//      4); the other FP8 kernels: 6;
//    - FP4 without a residual: 8.
static bool make_plan(int mode, int dt, bool res, bool w16, int hidden, const DeviceInfo& di,
                      Plan& pl)
{
    const int nv = hidden / elems_per_vec(dt);
    pl.mode = mode;
    pl.dt = dt;
    pl.res = res;
    const int forced = g_schedule.load();
    const long long stage = static_cast<long long>(nv) * 16 * (res ? 2 : 1);
    const int group = 16 / elems_per_vec(dt);

    // Row per warp: a warp holds the row in at most 8 vectors per lane (hidden <= 2048 for
    // 16-bit input) and each warp keeps its own two-row ring.
    const int warp_red = kRedFloatsWarp * 4;
    const bool warp_fits = nv <= 256 && 2 * stage + warp_red + 32 <= di.smem_optin;
    const bool warp_auto = res ? nv <= 64 : nv <= 256;
    if (warp_fits && (forced == SCHED_WARP || (forced == 0 && warp_auto))) {
        int vpt = 1;
        while (32 * vpt < nv) vpt *= 2;
        if (mode == MODE_NVFP4 && vpt < group) vpt = group;
        const int tv = g_tune_vpt.load();
        if (tv > vpt) vpt = tv;
        int warps = g_tune_warps.load();
        if (warps == 0) warps = 8;
        int stages = g_tune_stages.load();
        if (stages < 2) stages = 2;                 // automatic, or a single slot asked for
        auto bytes = [&](int w, int st) { return w * st * stage + warp_red + w * st * 16; };
        while (stages > 2 && bytes(warps, stages) > di.smem_optin) --stages;
        while (warps > 1 && bytes(warps, stages) > di.smem_optin) warps /= 2;
        pl.sched = SCHED_WARP;
        pl.vpt = vpt;
        pl.threads = 32 * warps;
        pl.stages = stages;
        pl.smem = static_cast<int>(bytes(warps, stages));
        pl.ctas_per_sm = g_tune_ctas.load();
        return true;
    }

    // A cluster of C CTAs per row: for rows whose two-slot ring does not fit one CTA's shared
    // memory or that need more than 512 threads (or when forced). The smallest C of 2, 4, 8, 16
    // whose slice slot holds at most 32 KB (64 KB for the one-slot FP8 kernels, below):
    // three CTAs per SM, so one CTA's row-end barrier and exchange overlap the others' work
    // (measured on GB300: 4.5-5.1 TB/s against 3.7-4.5 TB/s with one CTA per SM at 32768). Else
    // the smallest whose ring fits; slices hold whole FP4 scale blocks; 4 or 8 vectors per
    // thread (below).
    const int red_bytes = kRedFloats * 4;
    const bool pipe_fits = 2 * stage + red_bytes + 2 * 16 <= di.smem_optin;
    // A CTA covers at most 512 threads x 8 vectors: wider rows take a cluster even when two of
    // their ring slots would fit one CTA's shared memory (rows without a residual).
    const bool one_cta = pipe_fits && nv <= 512 * 8;
    if (forced == SCHED_CLUSTER || (!one_cta && forced != SCHED_REG)) {
        const int tune_c = g_tune_cluster.load();
        const int blk = mode == MODE_MXFP4 ? 32 : 16;
        // The FP8 kernels with two exchanges per row (a weight offset, or fp32 input) keep s in
        // registers, so their ring is one slot, refilled right after the first exchange; the
        // slot may then be twice as large, for half as many CTAs per row. Measured on GB300 (read
        // flush), against two slots on clusters twice as large:
        //  - fp16 with an offset, 4096 x 65536 + residual: 377 against 481 us (clusters of 4);
        //    2048 x 131072: 420 against 654 us (8); 8192 x 32768: 355 against 408 us (2);
        //    without a residual, 4096 x 65536: 334.5 against 349 us (2);
        //  - bf16 with an offset, 4096 x 65536: 435 against 556 us;
        //  - fp32, 2048 x 65536 + residual: 293 against 486 us (8 vectors per thread both);
        //    4096 x 32768: 264 against 334.5 us; without a residual, 238 against 245 us.
        const bool two_x = mode == MODE_FP8 && !w16;
        const long long small_slot = two_x ? 65536 : 32768;
        int best = 0;
        for (int c = 2; c <= 16; c *= 2) {
            if (tune_c != 0 && c != tune_c) continue;
            if (nv % c != 0) continue;
            const int nvc = nv / c;
            if (mode != MODE_FP8 && (nvc * elems_per_vec(dt)) % blk != 0) continue;
            const long long cstage = static_cast<long long>(nvc) * 16 * (res ? 2 : 1);
            if (2 * cstage + red_bytes + 2 * 16 + kClusterXchBytes > di.smem_optin) continue;
            if ((nvc + 7) / 8 > 512) continue;
            if (best == 0) best = c;              // smallest that fits
            if (cstage <= small_slot || tune_c != 0) {
                best = c;                         // smallest with a small slot
                break;
            }
        }
        const bool one_exchange = mode != MODE_FP8 || w16;
        if (best != 0) {
            const int nvc = nv / best;
            const long long cstage = static_cast<long long>(nvc) * 16 * (res ? 2 : 1);
            // Vectors per thread (instantiated for 4 and 8). FP8 and NVFP4: 8, so a CTA has half
            // the threads and twice as many fit an SM beside the others of their cluster.
            // Measured on GB300 against 4:
            //  - FP8 without a residual: 283 against 453 us at 2048 x 131072, 263 against 353 us
            //    at 4096 x 65536;
            //  - FP8 with a weight offset: 666 against 811 us at 2048 x 131072, 489 against
            //    507 us at 4096 x 65536;
            //  - clusters of 16 with a residual: FP8 470 against 488 us, NVFP4 314 against
            //    347 us (2048 x 131072);
            //  - fp32 input: FP8 at 2048 x 65536 486 against 689 us, 4096 x 32768 334.5 against
            //    400 us (two slots); NVFP4 at 2048 x 65536 322 against 339 us;
            //  - within 2 % of 4 on the other shapes, except the W16 FP8 kernel with a residual
            //    in clusters of 2 or 4, which keeps 4 (320 against 324 us at 8192 x 32768).
            // MXFP4: 4, or 8 when that would take more than 256 threads. 8 measured slower at
            // 2048 x 131072 bf16 (422 against 373 us) and at 4096 x 32768 fp32 (317 against
            // 298 us), faster only at 2048 x 65536 fp32 (412 against 450 us).
            int cv = g_tune_vpt.load();
            if (cv < 4 || (nvc + cv - 1) / cv > 512) {
                cv = 4;
                const int per = mode == MODE_FP8 ? 512 : 256;
                while (cv < 8 && nvc > per * cv) cv *= 2;
                const bool small_w16_res = mode == MODE_FP8 && w16 && res && best < 8;
                if ((mode == MODE_FP8 || mode == MODE_NVFP4) && !small_w16_res) cv = 8;
            }
            // ring slots, reduction area, per slot an mbarrier and a row number, exchange slots.
            // Kernels with one exchange per row (all but FP8 with an offset or fp32 input) hold
            // two rows while their exchange is in flight, so a third slot keeps a load going:
            // measured on GB300, 8-25 % faster than two slots at 16384-131072 elements.
            // With a residual those kernels split the slot: the ring holds x only and one more
            // slot holds the next row's residual (its mbarrier and row number one more entry),
            // which needs three ring slots at least.
            const bool split = one_exchange && res;
            // kernels with two exchanges refill their slot right after the first (s is then in
            // registers), so one slot is a valid ring for them
            const int min_stages = split ? 3 : one_exchange ? 2 : 1;
            int stages = g_tune_stages.load();
            if (stages == 0) stages = two_x ? 1 : one_exchange ? 3 : 2;
            if (stages < min_stages) stages = min_stages;
            auto cbytes = [&](int st) {
                return split ? st * (cstage / 2) + cstage / 2 + red_bytes + (st + 1) * 16 + kClusterXchBytes
                             : st * cstage + red_bytes + st * 16 + kClusterXchBytes;
            };
            while (stages > min_stages && cbytes(stages) > di.smem_optin) --stages;
            pl.sched = SCHED_CLUSTER;
            pl.cluster = best;
            pl.vpt = cv;
            pl.threads = ((nvc + cv - 1) / cv + 31) / 32 * 32;
            pl.stages = stages;
            pl.smem = static_cast<int>(cbytes(stages));
            pl.ctas_per_sm = 0;
            return true;
        }
    }

    int vpt = g_tune_vpt.load();
    if (vpt == 0) {
        if (mode != MODE_FP8 && mode != MODE_AMAX && res) {
            // FP4 with a residual (bandwidth-bound): ~128 threads for short rows, 256 at 4096,
            // 8 vectors per thread from 5120 on; MXFP4 rows of up to 256 vectors take one vector
            // per thread (measured on GB300 at 65536 x 2048: ncu DRAM throughput 83.7 % median,
            // 83.3 - 84.1 % over 5 launches, against 83.2 % with launches from 78.9 to 85.1 %
            // with two)
            vpt = 2;
            while (vpt < 8 && nv > 512 * vpt) vpt *= 2;
            if (mode == MODE_NVFP4 && nv <= 512) vpt = 4;
            if (mode == MODE_MXFP4 && nv <= 256) vpt = 1;
        } else {
            // the power of two nearest nv / 128 vectors per thread
            vpt = 1;
            while (vpt < 8 && 2 * nv > 3 * 128 * vpt) vpt *= 2;
            if (mode == MODE_FP8 && !w16 && vpt > 4) vpt = 4;
            if (mode == MODE_FP8 && nv <= 256) vpt = 4;
        }
        while (vpt < 8 && (nv + vpt - 1) / vpt > 512) vpt *= 2;
        // NVFP4 threads own whole 16-element scale blocks (2 vectors, 4 for fp32 input)
        if (mode == MODE_NVFP4 && vpt < group) vpt = group;
    }
    int threads = ((nv + vpt - 1) / vpt + 31) / 32 * 32;
    if (threads > 512) return false;
    pl.vpt = vpt;
    pl.threads = threads;

    pl.sched = (forced == SCHED_REG || !pipe_fits) ? SCHED_REG : SCHED_PIPE;
    pl.ctas_per_sm = g_tune_ctas.load();
    if (pl.ctas_per_sm == 0) {
        if (mode == MODE_FP8) pl.ctas_per_sm = nv <= 256 ? 384 / threads : (w16 ? 8 : 6);
        else if (!res) pl.ctas_per_sm = 8;
        else pl.ctas_per_sm = 8;
    }
    // The FP8 kernel with a weight offset and 16-bit input (four vectors per thread) keeps w in
    // a shared-memory table of 32 bytes per vector (at most 2048 vectors per row, so the table
    // and one slot always fit). Its ring takes two slots when that costs no resident CTA, else
    // one: measured on GB300, one slot is faster for rows of 4096 and 8192 (3 and 6 CTAs per SM
    // instead of 2 and 4) and two for rows of 2048 and 16384, where the CTA count is the same.
    const bool gamma_table = mode == MODE_FP8 && !w16 && dt != DT_F32 && vpt == 4 &&
                             pl.sched == SCHED_PIPE;
    if (gamma_table) {
        const long long table = 32LL * nv;
        auto bytes = [&](int st) { return st * stage + table + red_bytes + st * 16; };
        // resident CTAs: the CTA cap, the kernel's register cap in 256-register warp units, and
        // shared memory
        auto ctas = [&](int st) {
            long long c = pl.ctas_per_sm;
            constexpr int regs = reg_cap<DT_FP16, true, MODE_FP8, 4, SCHED_PIPE, false>();
            const long long by_regs = (65536 / (regs * 32)) / (threads / 32);
            const long long by_smem = di.smem_per_sm / (bytes(st) + di.smem_reserved);
            if (by_regs < c) c = by_regs;
            if (by_smem < c) c = by_smem;
            return c;
        };
        int stages = g_tune_stages.load();
        if (stages == 0) stages = (bytes(2) <= di.smem_optin && ctas(2) >= ctas(1)) ? 2 : 1;
        while (stages > 1 && bytes(stages) > di.smem_optin) --stages;
        pl.stages = stages;
        pl.smem = static_cast<int>(bytes(stages));
    } else if (pl.sched == SCHED_PIPE) {
        int stages = g_tune_stages.load();
        // kernels that keep s in the slot refill it at the end of the row: two slots at least
        if (stages == 1 && (mode != MODE_FP8 || w16)) stages = 2;
        if (stages == 0)
            stages = (mode != MODE_FP8 && res && nv >= 2048) ? 3 : 2;
        // ring slots, reduction area, then per slot an mbarrier and the slot's row number
        while (stages > 2 && stages * stage + red_bytes + stages * 16 > di.smem_optin) --stages;
        pl.stages = stages;
        pl.smem = static_cast<int>(stages * stage) + red_bytes + stages * 16;
    } else {
        pl.stages = 0;
        pl.smem = red_bytes;
    }
    return true;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks shared by every entry point. Returns RMSQ_OK with *empty set for a valid rows == 0
// call, whose data pointers are not examined.
static rmsq_status check_common(const void* input, const void* residual, const void* residual_output,
                                const void* gamma, int64_t rows, int64_t hidden, int dtype,
                                float epsilon, float weight_offset, int min_multiple, bool* empty)
{
    *empty = false;
    if (dtype != RMSQ_BF16 && dtype != RMSQ_FP16 && dtype != RMSQ_F32) return RMSQ_ERR_DTYPE;
    const int64_t max_h = dtype == RMSQ_F32 ? RMSQ_MAX_HIDDEN / 2 : RMSQ_MAX_HIDDEN;
    const int64_t one_cta = dtype == RMSQ_F32 ? RMSQ_ONE_CTA_HIDDEN / 2 : RMSQ_ONE_CTA_HIDDEN;
    if (rows < 0 || hidden < min_multiple || hidden > max_h || hidden % min_multiple != 0)
        return RMSQ_ERR_SHAPE;
    if (hidden > one_cta && hidden % 256 != 0) return RMSQ_ERR_SHAPE;   // cluster slices
    if (!(epsilon >= 0.0f) || !std::isfinite(epsilon) || !std::isfinite(weight_offset))
        return RMSQ_ERR_VALUE;
    if (rows == 0) {
        *empty = true;
        return RMSQ_OK;
    }
    if (!input || !gamma) return RMSQ_ERR_NULL;
    if ((residual == nullptr) != (residual_output == nullptr)) return RMSQ_ERR_NULL;
    if (!aligned16(input) || !aligned16(gamma) || !aligned16(residual) || !aligned16(residual_output))
        return RMSQ_ERR_ALIGN;
    return RMSQ_OK;
}

static Params base_params(const void* input, const void* residual, void* residual_output,
                          const void* gamma, int64_t rows, int64_t hidden, int dtype, float epsilon,
                          float weight_offset, const DeviceInfo& di)
{
    Params p;
    std::memset(&p, 0, sizeof p);
    p.x = input;
    p.res = residual;
    p.res_out = residual_output;
    p.gamma = gamma;
    p.err = di.err;
    p.rows = rows;
    p.hidden = static_cast<int>(hidden);
    p.nvec = static_cast<int>(hidden / elems_per_vec(dtype));
    p.eps = epsilon;
    p.offset = weight_offset;
    p.timeout_ns = g_timeout_ns.load();
    return p;
}

static rmsq_status launch(int mode, Params& p, bool res, int dtype, const DeviceInfo& di,
                          cudaStream_t stream)
{
    Plan pl;
    const bool w16 = dtype != DT_F32 && p.offset == 0.0f;
    if (!make_plan(mode, dtype, res, w16, p.hidden, di, pl)) return RMSQ_ERR_SHAPE;
    pl.w16 = w16;
    p.stages = pl.stages;
    cudaError_t e;
    switch (mode) {
    case MODE_FP8: e = dispatch_fp8(pl, p, stream); break;
    case MODE_NVFP4: e = dispatch_nvfp4(pl, p, stream); break;
    case MODE_MXFP4: e = dispatch_mxfp4(pl, p, stream); break;
    default: e = dispatch_amax(pl, p, stream); break;
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return RMSQ_ERR_LAUNCH;
    }
    return RMSQ_OK;
}

// ------------------------------------------------------------------------------------------
// Diagnostic kernels
// ------------------------------------------------------------------------------------------

__global__ void selftest_wait_kernel(unsigned int* err, unsigned long long timeout_ns)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    // Nothing arrives on this barrier: the wait must run out and report it.
    const bool ok = mbar_wait_bounded(smem_u32(&bar), 0, timeout_ns);
    if (__syncthreads_or(!ok) && threadIdx.x == 0) atomicOr(err, ERRF_WAIT_TIMEOUT);
}

__global__ void debug_convert_kernel(int fmt, const float* __restrict__ in,
                                     unsigned char* __restrict__ out, long long n)
{
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const float v = in[i];
        if (fmt == 0) {
            out[i] = static_cast<unsigned char>(cvt_e4m3x2(v, 0.0f) & 0xFFu);
        } else {
            const float q[4] = {v, 0.0f, 0.0f, 0.0f};
            out[i] = static_cast<unsigned char>(cvt_e2m1x4(q) & 0xFu);
        }
    }
}

// The global scale of a tensor with no rows (max |y| = 0): 1.
__global__ void global_scale_of_empty_kernel(float* gs) { *gs = 1.0f; }

}  // namespace rmsq

using namespace rmsq;

// ------------------------------------------------------------------------------------------
// C ABI
// ------------------------------------------------------------------------------------------

extern "C" rmsq_status rmsnorm_quant_fp8(const void* input, const void* residual,
                                         void* residual_output, const void* gamma, int64_t rows,
                                         int64_t hidden, int dtype, float epsilon,
                                         float weight_offset, float scale_ub, void* output,
                                         void* scale_output, int scale_dtype, void* stream)
{
    bool empty;
    rmsq_status st = check_common(input, residual, residual_output, gamma, rows, hidden, dtype,
                                  epsilon, weight_offset, dtype == RMSQ_F32 ? 4 : 8, &empty);
    if (st != RMSQ_OK) return st;
    if (scale_dtype != RMSQ_F32 && scale_dtype != RMSQ_BF16 && scale_dtype != RMSQ_FP16)
        return RMSQ_ERR_DTYPE;
    if (!(scale_ub > 0.0f)) return RMSQ_ERR_VALUE;
    if (empty) return RMSQ_OK;
    if (!output || !scale_output) return RMSQ_ERR_NULL;
    if (!aligned16(output) || !aligned16(scale_output)) return RMSQ_ERR_ALIGN;
    const DeviceInfo* di = device_info();
    if (!di) return RMSQ_ERR_DEVICE;
    Params p = base_params(input, residual, residual_output, gamma, rows, hidden, dtype, epsilon,
                           weight_offset, *di);
    p.out = output;
    p.scale_out = scale_output;
    p.scale_ub = scale_ub;
    p.scale_dtype = scale_dtype;
    return launch(MODE_FP8, p, residual != nullptr, dtype, *di, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------------------------------
// rmsnorm_quant_fp8_static_scratch: the FP8 call with its scratch in a file-scope array
// ------------------------------------------------------------------------------------------

// The FP8 kernel's only scratch is the 32-bit counter that hands out the last rows of a launch.
// For callers that must know every byte of device memory the library touches, this entry point
// keeps that counter in its own 256-byte array, reserved on every device that loads the library
// until the process exits, and clears it on the caller's stream before each launch.
constexpr int kStaticScratchWords = 64;
static __device__ __align__(256) unsigned int g_fp8_static_scratch[kStaticScratchWords];
static unsigned int* g_fp8_static_scratch_addr[kMaxDevices];   // its device address, per device

extern "C" rmsq_status rmsnorm_quant_fp8_static_scratch(
    const void* input, const void* residual, void* residual_output, const void* gamma,
    int64_t rows, int64_t hidden, int dtype, float epsilon, float weight_offset, float scale_ub,
    void* output, void* scale_output, int scale_dtype, void* stream)
{
    bool empty;
    rmsq_status st = check_common(input, residual, residual_output, gamma, rows, hidden, dtype,
                                  epsilon, weight_offset, dtype == RMSQ_F32 ? 4 : 8, &empty);
    if (st != RMSQ_OK) return st;
    if (scale_dtype != RMSQ_F32 && scale_dtype != RMSQ_BF16 && scale_dtype != RMSQ_FP16)
        return RMSQ_ERR_DTYPE;
    if (!(scale_ub > 0.0f)) return RMSQ_ERR_VALUE;
    if (rows > INT32_MAX) return RMSQ_ERR_SHAPE;   // beyond what the 32-bit counter can hand out
    if (empty) return RMSQ_OK;
    if (!output || !scale_output) return RMSQ_ERR_NULL;
    if (!aligned16(output) || !aligned16(scale_output)) return RMSQ_ERR_ALIGN;
    const DeviceInfo* di = device_info();
    if (!di) return RMSQ_ERR_DEVICE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return RMSQ_ERR_DEVICE;
    }
    unsigned int* scratch = nullptr;
    {
        // first call on this device: look up the array's device address (the name alone is a
        // host-side stand-in, not an address a kernel can use)
        std::lock_guard<std::mutex> lock(g_mu);
        if (g_fp8_static_scratch_addr[dev] == nullptr) {
            void* addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_fp8_static_scratch) != cudaSuccess || addr == nullptr) {
                cudaGetLastError();
                return RMSQ_ERR_DEVICE;
            }
            g_fp8_static_scratch_addr[dev] = static_cast<unsigned int*>(addr);
        }
        scratch = g_fp8_static_scratch_addr[dev];
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the counter must start at zero; the last call may have left anything in it
    if (cudaMemsetAsync(scratch, 0, sizeof(unsigned int) * kStaticScratchWords, s) != cudaSuccess) {
        cudaGetLastError();
        return RMSQ_ERR_LAUNCH;
    }
    Params p = base_params(input, residual, residual_output, gamma, rows, hidden, dtype, epsilon,
                           weight_offset, *di);
    p.out = output;
    p.scale_out = scale_output;
    p.scale_ub = scale_ub;
    p.scale_dtype = scale_dtype;
    p.rowctr = scratch;
    return launch(MODE_FP8, p, residual != nullptr, dtype, *di, s);
}

static rmsq_status fp4_common(int mode, const void* input, const void* residual,
                              void* residual_output, const void* gamma, int64_t rows,
                              int64_t hidden, int dtype, float epsilon, float weight_offset,
                              const float* global_scale, void* output, void* block_scale,
                              int scale_layout, void* stream)
{
    const int block = mode == MODE_NVFP4 ? 16 : 32;
    bool empty;
    rmsq_status st = check_common(input, residual, residual_output, gamma, rows, hidden, dtype,
                                  epsilon, weight_offset, block, &empty);
    if (st != RMSQ_OK) return st;
    if (scale_layout != RMSQ_SCALE_ROW_MAJOR && scale_layout != RMSQ_SCALE_SWIZZLED_128x4)
        return RMSQ_ERR_DTYPE;
    if (empty) return RMSQ_OK;
    if (!output || !block_scale) return RMSQ_ERR_NULL;
    if (mode == MODE_NVFP4 && !global_scale) return RMSQ_ERR_NULL;
    if (!aligned16(output) || !aligned16(block_scale)) return RMSQ_ERR_ALIGN;
    if (mode == MODE_NVFP4 && (reinterpret_cast<uintptr_t>(global_scale) & 3u)) return RMSQ_ERR_ALIGN;
    const DeviceInfo* di = device_info();
    if (!di) return RMSQ_ERR_DEVICE;
    Params p = base_params(input, residual, residual_output, gamma, rows, hidden, dtype, epsilon,
                           weight_offset, *di);
    p.out = output;
    p.scale_out = block_scale;
    p.gs = global_scale;
    p.swizzled = scale_layout == RMSQ_SCALE_SWIZZLED_128x4;
    p.nsf = static_cast<int>(hidden / block);
    p.k_tiles = (p.nsf + 3) / 4;
    return launch(mode, p, residual != nullptr, dtype, *di, static_cast<cudaStream_t>(stream));
}

extern "C" rmsq_status rmsnorm_quant_nvfp4(const void* input, const void* residual,
                                           void* residual_output, const void* gamma, int64_t rows,
                                           int64_t hidden, int dtype, float epsilon,
                                           float weight_offset, const float* global_scale,
                                           void* output, void* block_scale, int scale_layout,
                                           void* stream)
{
    return fp4_common(MODE_NVFP4, input, residual, residual_output, gamma, rows, hidden, dtype,
                      epsilon, weight_offset, global_scale, output, block_scale, scale_layout,
                      stream);
}

extern "C" rmsq_status rmsnorm_quant_mxfp4(const void* input, const void* residual,
                                           void* residual_output, const void* gamma, int64_t rows,
                                           int64_t hidden, int dtype, float epsilon,
                                           float weight_offset, void* output, void* block_scale,
                                           int scale_layout, void* stream)
{
    return fp4_common(MODE_MXFP4, input, residual, residual_output, gamma, rows, hidden, dtype,
                      epsilon, weight_offset, nullptr, output, block_scale, scale_layout, stream);
}

extern "C" rmsq_status rmsnorm_nvfp4_global_scale(const void* input, const void* residual,
                                                  const void* gamma, int64_t rows, int64_t hidden,
                                                  int dtype, float epsilon, float weight_offset,
                                                  float* gs_out, void* stream)
{
    if (!gs_out) return RMSQ_ERR_NULL;
    // the residual is read but no residual_output is written: pass it as its own pair partner
    bool empty;
    rmsq_status st = check_common(input, residual, residual, gamma, rows, hidden, dtype, epsilon,
                                  weight_offset, 16, &empty);
    if (st != RMSQ_OK) return st;
    if (reinterpret_cast<uintptr_t>(gs_out) & 3u) return RMSQ_ERR_ALIGN;
    const DeviceInfo* di = device_info();
    if (!di) return RMSQ_ERR_DEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (rows > 0) {
        // one launch: its last CTA writes gs (the kernel's epilogue)
        Params p = base_params(input, residual, nullptr, gamma, rows, hidden, dtype, epsilon,
                               weight_offset, *di);
        p.scale_out = gs_out;
        return launch(MODE_AMAX, p, residual != nullptr, dtype, *di, s);
    }
    // no rows: an all-zero tensor's gs, 1
    global_scale_of_empty_kernel<<<1, 1, 0, s>>>(gs_out);
    if (cudaGetLastError() != cudaSuccess) return RMSQ_ERR_LAUNCH;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return RMSQ_OK;
}

extern "C" const char* rmsq_status_string(rmsq_status status)
{
    switch (status) {
    case RMSQ_OK: return "RMSQ_OK";
    case RMSQ_ERR_NULL: return "RMSQ_ERR_NULL: a required pointer is NULL or residual pointers are unpaired";
    case RMSQ_ERR_SHAPE: return "RMSQ_ERR_SHAPE: rows or hidden out of range, or hidden not a multiple of the block";
    case RMSQ_ERR_ALIGN: return "RMSQ_ERR_ALIGN: a data pointer is not 16-byte aligned";
    case RMSQ_ERR_DTYPE: return "RMSQ_ERR_DTYPE: unknown dtype, scale dtype or scale layout";
    case RMSQ_ERR_LAUNCH: return "RMSQ_ERR_LAUNCH: the CUDA launch failed";
    case RMSQ_ERR_VALUE: return "RMSQ_ERR_VALUE: epsilon, weight_offset or scale_ub out of range";
    case RMSQ_ERR_DEVICE: return "RMSQ_ERR_DEVICE: no usable compute capability 10.3 device";
    case RMSQ_ERR_TIMEOUT: return "RMSQ_ERR_TIMEOUT: a bounded device-side wait ran out";
    }
    return "RMSQ_UNKNOWN_STATUS";
}

extern "C" rmsq_status rmsq_device_status(void)
{
    const DeviceInfo* di = device_info();
    if (!di) return RMSQ_ERR_DEVICE;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return RMSQ_ERR_LAUNCH;
    }
    unsigned int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_err_word, sizeof word) != cudaSuccess) {
        cudaGetLastError();
        return RMSQ_ERR_LAUNCH;
    }
    if (word != 0) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_err_word, &zero, sizeof zero);
        cudaMemset(di->counters, 0, sizeof(unsigned int) * kCounterSlots * 8);
        return RMSQ_ERR_TIMEOUT;
    }
    return RMSQ_OK;
}

extern "C" int rmsq_set_schedule(int schedule)
{
    if (schedule < 0 || schedule > 4) schedule = 0;
    return g_schedule.exchange(schedule);
}

extern "C" rmsq_status rmsq_set_tuning(int stages, int ctas_per_sm, int vectors_per_thread)
{
    if (stages < 0 || stages > 8 || ctas_per_sm < 0 || ctas_per_sm > 32 ||
        (vectors_per_thread != 0 && vectors_per_thread != 1 && vectors_per_thread != 2 &&
         vectors_per_thread != 4 && vectors_per_thread != 8))
        return RMSQ_ERR_VALUE;
    g_tune_stages = stages;
    g_tune_ctas = ctas_per_sm;
    g_tune_vpt = vectors_per_thread;
    return RMSQ_OK;
}

extern "C" rmsq_status rmsq_set_row_warps(int warps_per_cta)
{
    if (warps_per_cta < 0 || warps_per_cta > 16) return RMSQ_ERR_VALUE;
    g_tune_warps = warps_per_cta;
    return RMSQ_OK;
}

extern "C" rmsq_status rmsq_set_cluster_size(int ctas_per_cluster)
{
    if (ctas_per_cluster != 0 && ctas_per_cluster != 2 && ctas_per_cluster != 4 &&
        ctas_per_cluster != 8 && ctas_per_cluster != 16)
        return RMSQ_ERR_VALUE;
    g_tune_cluster = ctas_per_cluster;
    return RMSQ_OK;
}

extern "C" int rmsq_set_dynamic_rows(int enable)
{
    return g_dynamic_rows.exchange(enable != 0) ? 1 : 0;
}

extern "C" int rmsq_set_pdl(int enable)
{
    return g_pdl.exchange(enable != 0) ? 1 : 0;
}

extern "C" void rmsq_set_wait_timeout_ns(uint64_t timeout_ns)
{
    g_timeout_ns = timeout_ns > 0 ? timeout_ns : 1;
}

extern "C" rmsq_status rmsq_selftest_wait_timeout(uint64_t timeout_ns, void* stream)
{
    const DeviceInfo* di = device_info();
    if (!di) return RMSQ_ERR_DEVICE;
    if (timeout_ns > 10000000000ull) return RMSQ_ERR_VALUE;
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(di->err, timeout_ns);
    if (cudaGetLastError() != cudaSuccess) return RMSQ_ERR_LAUNCH;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return RMSQ_OK;
}

extern "C" rmsq_status rmsq_debug_convert(int fmt, const float* in, uint8_t* out, int64_t n,
                                          void* stream)
{
    if (!in || !out) return RMSQ_ERR_NULL;
    if (fmt != 0 && fmt != 1) return RMSQ_ERR_DTYPE;
    if (n < 0) return RMSQ_ERR_SHAPE;
    if (n == 0) return RMSQ_OK;
    const DeviceInfo* di = device_info();
    if (!di) return RMSQ_ERR_DEVICE;
    long long blocks = (n + 255) / 256;
    if (blocks > 8LL * di->sms * 8) blocks = 8LL * di->sms * 8;
    debug_convert_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        fmt, in, out, n);
    if (cudaGetLastError() != cudaSuccess) return RMSQ_ERR_LAUNCH;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return RMSQ_OK;
}

extern "C" uint64_t rmsq_launch_count(void) { return g_launches.load(); }

extern "C" rmsq_status rmsq_plan(int mode, int dtype, int residual, float weight_offset,
                                 int64_t hidden, int smem_optin, int smem_per_sm, int smem_reserved,
                                 rmsq_plan_info* out)
{
    if (!out) return RMSQ_ERR_NULL;
    if (mode < MODE_FP8 || mode > MODE_AMAX) return RMSQ_ERR_VALUE;
    // the entry point's own checks of dtype, width and weight_offset (rows = 0: no pointers)
    const int min_multiple = mode == MODE_FP8 ? (dtype == RMSQ_F32 ? 4 : 8)
                             : mode == MODE_MXFP4 ? 32 : 16;
    bool empty;
    rmsq_status st = check_common(nullptr, nullptr, nullptr, nullptr, 0, hidden, dtype, 0.0f,
                                  weight_offset, min_multiple, &empty);
    if (st != RMSQ_OK) return st;
    DeviceInfo di;
    if (smem_optin == 0) {
        const DeviceInfo* cur = device_info();
        if (!cur) return RMSQ_ERR_DEVICE;
        di = *cur;
    } else {
        if (smem_optin < 0 || smem_per_sm < smem_optin || smem_reserved < 0) return RMSQ_ERR_VALUE;
        di.smem_optin = smem_optin;
        di.smem_per_sm = smem_per_sm;
        di.smem_reserved = smem_reserved;
    }
    Plan pl;
    const bool w16 = dtype != DT_F32 && weight_offset == 0.0f;
    if (!make_plan(mode, dtype, residual != 0, w16, static_cast<int>(hidden), di, pl))
        return RMSQ_ERR_SHAPE;
    out->schedule = pl.sched;
    out->vectors_per_thread = pl.vpt;
    out->threads = pl.threads;
    out->stages = pl.stages;
    out->cluster = pl.sched == SCHED_CLUSTER ? pl.cluster : 1;
    out->smem_bytes = pl.smem;
    out->ctas_per_sm = pl.ctas_per_sm;
    out->w16 = w16 ? 1 : 0;
    return RMSQ_OK;
}
