/*
 * rmsq.h -- C ABI of the GB300 (sm_103a) fused residual-add + RMSNorm + dynamic quantisation
 * library (librmsq.so).
 *
 * For each row r of a row-major [rows x hidden] activation the library computes, in one pass
 * over HBM:
 *
 *   s_i  = RN_dtype(input_i + residual_i)      written to residual_output ("pre-norm sum"),
 *                                              or s = input when there is no residual
 *   rstd = 1 / sqrt(sum_i s_i^2 / hidden + epsilon)                       (fp32 accumulation)
 *   y_i  = s_i * rstd * (gamma_i + weight_offset)                          (fp32)
 *
 * and quantises y in one of three ways:
 *
 *   FP8    amax = max_i |y_i|;  scale = min(amax, scale_ub) / 448;  q_i = E4M3(y_i / scale)
 *          -- Modular Mojo API docs, "rms_norm_fused_fp8" (arguments gamma, epsilon,
 *          weight_offset, scale_ub, scale_output) and "allreduce_residual_rmsnorm_fp8"
 *          (residual, residual_output; weight_offset "additive offset for gamma weights";
 *          scale_ub "upper bound for FP8 scale clamping").
 *   NVFP4  per 16 elements: s_b = E4M3(min(gs * amax_b / 6, 448));
 *          q_i = E2M1(y_i * gs / s_b), two codes per byte, element 2k in the low nibble
 *          -- FlashInfer "cute_dsl/rmsnorm_fp4quant.py", RMSNormFP4QuantKernel phase 3
 *          (E4M3 scale format, block 16) and cvt_e2m1x8_f32.
 *   MXFP4  per 32 elements: e_b = clamp(ceil(log2(amax_b / 6)) + 127, 0, 255) (UE8M0);
 *          q_i = E2M1(y_i * 2^(127 - e_b)), and q = 0 for a block with e_b = 0
 *          -- the same file, phase 3 with the UE8M0 scale format (block 32),
 *          cvt_f32_to_ue8m0 and ue8m0_to_output_scale.
 *
 * All E4M3 / E2M1 conversions round to nearest even and saturate finite values ("satfinite").
 * A row whose FP8 scale is 0 (an all-zero y) gets codes 0 and scale 0.
 *
 * Conventions shared by every entry point below:
 *   - Every data pointer is caller-owned DEVICE memory of the current CUDA device, contiguous and
 *     row-major, and must be 16-byte aligned (RMSQ_ERR_ALIGN otherwise). The library never
 *     allocates, frees or synchronises; work is queued on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and the call returns at once.
 *   - rows == 0 is a valid empty call: nothing is launched, RMSQ_OK is returned and the data
 *     pointers are not examined (they may be NULL).
 *   - Arguments are checked on the host before anything is launched; on an error nothing is
 *     launched and no output is touched.
 *   - residual and residual_output are both NULL (no residual) or both non-NULL.
 *   - Inputs must be finite; NaN / Inf inputs give unspecified codes.
 *   - Calls on one stream are ordered; outputs of concurrent calls must not overlap.
 */
#ifndef RMSQ_H
#define RMSQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of input, residual, residual_output and gamma (one type for all four), and of an
 * FP8 scale_output. The pages list float32, float16 and bfloat16 ("rms_norm_fused_fp8",
 * parameters in_dtype and scales_dtype). */
typedef enum { RMSQ_BF16 = 0, RMSQ_FP16 = 1, RMSQ_F32 = 2 } rmsq_dtype;

/* Layout of an NVFP4 / MXFP4 block-scale tensor ("rmsnorm_fp4quant", argument
 * is_sf_swizzled_layout):
 *   RMSQ_SCALE_ROW_MAJOR       [rows][hidden / block], one byte each.
 *   RMSQ_SCALE_SWIZZLED_128x4  tiles of 128 rows x 4 scales, 512 bytes each, in the order
 *                              [row / 128][sf / 4][row % 32][(row % 128) / 32][sf % 4], with the
 *                              number of 4-scale tiles per row rounded up; the tensor holds
 *                              ceil(rows / 128) * ceil(hidden / block / 4) * 512 bytes. Bytes of
 *                              the padding (rows past `rows`, scales past hidden / block) are not
 *                              written. */
typedef enum { RMSQ_SCALE_ROW_MAJOR = 0, RMSQ_SCALE_SWIZZLED_128x4 = 1 } rmsq_scale_layout;

typedef enum {
    RMSQ_OK = 0,
    RMSQ_ERR_NULL = 1,    /* a required pointer is NULL, or only one of residual /
                             residual_output is given */
    RMSQ_ERR_SHAPE = 2,   /* rows < 0, or hidden outside [block, RMSQ_MAX_HIDDEN] or not a
                             multiple of the mode's block (FP8: 8 elements for 16-bit types and
                             4 for fp32; NVFP4: 16; MXFP4: 32), or a row wider than
                             RMSQ_ONE_CTA_HIDDEN that is not a multiple of 256 elements */
    RMSQ_ERR_ALIGN = 3,   /* a data pointer is not 16-byte aligned */
    RMSQ_ERR_DTYPE = 4,   /* unknown rmsq_dtype, scale dtype or scale layout */
    RMSQ_ERR_LAUNCH = 5,  /* the CUDA launch failed (cudaGetLastError after launch) */
    RMSQ_ERR_VALUE = 6,   /* epsilon < 0 or not finite, scale_ub <= 0 or NaN, or a weight_offset
                             that is not finite */
    RMSQ_ERR_DEVICE = 7,  /* no usable CUDA device, or the device is not compute capability 10.3 */
    RMSQ_ERR_TIMEOUT = 8  /* reported by rmsq_device_status: a bounded device-side wait ran out */
} rmsq_status;

/* Largest hidden size any entry point accepts, in elements (fp32 input: half of it). Rows wider
 * than RMSQ_ONE_CTA_HIDDEN (fp32: half of it) are split over a thread-block cluster of up to 16
 * CTAs and must be a multiple of 256 elements. */
#define RMSQ_MAX_HIDDEN 131072
#define RMSQ_ONE_CTA_HIDDEN 32768

/* ---------------------------------------------------------------------------------------------
 * rmsnorm_quant_fp8 -- residual add + RMSNorm + FP8 E4M3 with a per-row dynamic scale.
 * Follows "rms_norm_fused_fp8" (shape, output, gamma, epsilon, weight_offset, scale_ub,
 * scale_output) and, at one GPU, "allreduce_residual_rmsnorm_fp8" (residual, residual_output).
 *
 *   input            [rows x hidden] of `dtype`
 *   residual         [rows x hidden] of `dtype`, or NULL
 *   residual_output  [rows x hidden] of `dtype` receives s = RN_dtype(input + residual), or NULL
 *   gamma            [hidden] of `dtype`
 *   epsilon          added to the mean square (fp32)
 *   weight_offset    added to gamma in fp32 before the multiply (1.0 for Gemma-style weights)
 *   scale_ub         upper bound applied to the row amax before the scale is formed
 *   output           [rows x hidden] bytes, float8_e4m3fn codes
 *   scale_output     [rows] of `scale_dtype` (RMSQ_F32, RMSQ_BF16 or RMSQ_FP16): the row scale,
 *                    so that y ~= decode(q) * scale. A bf16 / fp16 scale is the fp32 scale
 *                    rounded to that type, and the codes are formed against the rounded value.
 * ------------------------------------------------------------------------------------------- */
rmsq_status rmsnorm_quant_fp8(const void* input, const void* residual, void* residual_output,
                              const void* gamma, int64_t rows, int64_t hidden, int dtype,
                              float epsilon, float weight_offset, float scale_ub, void* output,
                              void* scale_output, int scale_dtype, void* stream);

/* ---------------------------------------------------------------------------------------------
 * rmsnorm_quant_nvfp4 -- residual add + RMSNorm + NVFP4 (E2M1 with an E4M3 scale per 16
 * elements under an fp32 global scale). Follows "rmsnorm_fp4quant" (input, weight, y_fp4,
 * block_scale, global_scale, eps, block_size = 16, is_sf_swizzled_layout) plus the residual pair.
 *
 *   global_scale     DEVICE pointer to one fp32 gs, read by the kernel (so a captured CUDA graph
 *                    sees the value current at replay). gs multiplies the block scale and the
 *                    element factor: y ~= decode(q) * decode(s_b) / gs.
 *   output           [rows x hidden / 2] bytes, two E2M1 codes per byte (element 2k low nibble)
 *   block_scale      E4M3 codes in `scale_layout`
 * Other arguments as for rmsnorm_quant_fp8.
 * ------------------------------------------------------------------------------------------- */
rmsq_status rmsnorm_quant_nvfp4(const void* input, const void* residual, void* residual_output,
                                const void* gamma, int64_t rows, int64_t hidden, int dtype,
                                float epsilon, float weight_offset, const float* global_scale,
                                void* output, void* block_scale, int scale_layout, void* stream);

/* ---------------------------------------------------------------------------------------------
 * rmsnorm_quant_mxfp4 -- residual add + RMSNorm + MXFP4 (E2M1 with a UE8M0 power-of-two scale
 * per 32 elements, no global scale). Follows "rmsnorm_fp4quant" with block_size = 32.
 *
 *   output           [rows x hidden / 2] bytes, two E2M1 codes per byte (element 2k low nibble)
 *   block_scale      UE8M0 codes (scale = 2^(code - 127)) in `scale_layout`
 * Other arguments as for rmsnorm_quant_fp8.
 * ------------------------------------------------------------------------------------------- */
rmsq_status rmsnorm_quant_mxfp4(const void* input, const void* residual, void* residual_output,
                                const void* gamma, int64_t rows, int64_t hidden, int dtype,
                                float epsilon, float weight_offset, void* output,
                                void* block_scale, int scale_layout, void* stream);

/* ---------------------------------------------------------------------------------------------
 * rmsnorm_nvfp4_global_scale -- the device-side pre-pass that forms the NVFP4 global scale
 * gs = 448 * 6 / max_{r,i} |y_ri| over the whole tensor, so that the largest block scale lands on
 * the largest E4M3 value ("rmsnorm_fp4quant" takes gs as a precomputed [1] fp32 tensor; this is
 * the step that precomputes it). Reads input (and residual) once more; writes nothing but the one
 * float. gs_out is a DEVICE pointer to one fp32; an all-zero tensor (or rows = 0) gives gs = 1.
 * One kernel launch: its last CTA turns the launch's running maximum into gs, using two words of
 * a per-launch slot of the library's scratch pool (4096 slots, taken in turn, left at zero), so
 * launches on different streams that run at the same time stay apart unless 4096 launches apart.
 * Arguments as for rmsnorm_quant_nvfp4 (no outputs besides gs_out).
 * ------------------------------------------------------------------------------------------- */
rmsq_status rmsnorm_nvfp4_global_scale(const void* input, const void* residual,
                                       const void* gamma, int64_t rows, int64_t hidden, int dtype,
                                       float epsilon, float weight_offset, float* gs_out,
                                       void* stream);

/* ---------------------------------------------------------------------------------------------
 * rmsnorm_quant_fp8_static_scratch -- rmsnorm_quant_fp8 with its scratch in a fixed array.
 * The pages have no counterpart: this is an addition for callers that cannot have a library
 * allocate or hand out device memory on their behalf, for example a runtime that reserves all
 * device memory itself before it starts serving, or a host thread that may not call the CUDA
 * allocator. Arguments, layouts, results and errors are those of rmsnorm_quant_fp8 (bit for bit
 * the same outputs), with these differences:
 *   - The only scratch the kernel uses, the counter that hands out the last rows of a launch,
 *     lives in a 256-byte array of this library's device memory, reserved on every GPU that
 *     loads the library until the process exits. The call allocates and frees nothing.
 *   - It clears that counter on `stream` before each launch. Every call shares the array, so
 *     calls that overlap on the GPU (other streams, other host threads) race and can hand out
 *     rows twice or not at all; order them on one stream.
 *   - rows above 2^31 - 1 (what the 32-bit counter can hand out) return RMSQ_ERR_SHAPE.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress) and
 *     returns RMSQ_ERR_DEVICE if that fails; make that first call before any stream capture.
 * ------------------------------------------------------------------------------------------- */
rmsq_status rmsnorm_quant_fp8_static_scratch(const void* input, const void* residual,
                                             void* residual_output, const void* gamma,
                                             int64_t rows, int64_t hidden, int dtype,
                                             float epsilon, float weight_offset, float scale_ub,
                                             void* output, void* scale_output, int scale_dtype,
                                             void* stream);

/* Human-readable name of a status code (static storage; never NULL). */
const char* rmsq_status_string(rmsq_status status);

/* ---------------------------------------------------------------------------------------------
 * rmsq_device_status -- errors raised on the device since the last call, for the current device.
 * Every wait inside a kernel on a bulk-copy (mbarrier) phase is bounded in time; a wait that runs
 * out sets a flag and the CTA stops, after waiting (for four times the bound) for the copies it
 * has in flight. After RMSQ_ERR_TIMEOUT the outputs of the launches since the last call are not
 * to be trusted. If one of those drain waits ran out as well (a second flag, reported the same
 * way), a CTA may have exited with a copy into its shared memory still pending; treat the CUDA
 * context as unreliable then. The cluster barrier of the cluster schedule is a hardware barrier
 * that cannot be bounded: every CTA of a cluster makes the same barrier calls (a timed-out wait
 * is shared through the cluster exchange and all CTAs stop together), so none is left waiting.
 * This call synchronises the device, returns RMSQ_ERR_TIMEOUT if a flag was set (RMSQ_OK
 * otherwise) and clears the flags, together with the scratch words (row counters, the
 * global-scale pre-pass's maximum) a stopped launch may have left behind.
 * ------------------------------------------------------------------------------------------- */
rmsq_status rmsq_device_status(void);

/* ---------------------------------------------------------------------------------------------
 * Tuning and diagnostics. None of these is needed for normal use.
 *
 * rmsq_set_schedule  forces the kernel schedule of later calls in this process: 0 = automatic,
 *                    1 = bulk-copy pipeline (rows staged in shared memory by the TMA engine, a
 *                    CTA per row), 2 = register-staged rows, 3 = row per warp (each warp owns
 *                    whole rows with its own bulk-copy ring; rows up to 256 vectors of 16 bytes,
 *                    i.e. hidden <= 2048 for 16-bit input), 4 = a thread-block cluster per row
 *                    (each CTA takes a slice through its own ring; the slices' sums meet in
 *                    distributed shared memory). Returns the previous value. A forced schedule
 *                    that does not fit the row falls back to the automatic choice.
 * rmsq_set_tuning    overrides the pipeline depth (stages, 0 = automatic, at most 8), CTAs per
 *                    SM (0 = automatic, at most 32) and vectors of 16 bytes per thread per row
 *                    (0 = automatic; 1, 2, 4 or 8). One stage is honoured by the kernels that
 *                    refill their slot before the row ends (FP8 with a weight offset or fp32
 *                    input, whose s is then held in registers); the others take their minimum of
 *                    two (three for the pipelined cluster kernels with a residual). Returns
 *                    RMSQ_ERR_VALUE for values out of range; a setting that needs more than 512
 *                    threads per CTA makes later calls fail with RMSQ_ERR_SHAPE.
 * rmsq_set_row_warps  warps per CTA of the row-per-warp schedule (0 = automatic, at most 16).
 *                    Returns RMSQ_ERR_VALUE out of range.
 * rmsq_set_cluster_size  CTAs per cluster of the cluster schedule (0 = automatic, else 2, 4, 8
 *                    or 16); the schedule itself is forced with rmsq_set_schedule(4). Returns
 *                    RMSQ_ERR_VALUE for other values.
 * rmsq_set_dynamic_rows  the CTA-per-row schedule hands the last quarter of its rows out one at a
 *                    time from a per-launch counter in the library's device memory, so CTAs on
 *                    SMs that get more HBM bandwidth take more rows (default). 0 deals every row
 *                    out round-robin. Returns the previous setting.
 * rmsq_set_pdl      kernels are launched with programmatic dependent launch by default (a
 *                    launch may be scheduled while the previous kernel on the stream finishes; it
 *                    waits for that kernel before touching global memory). 0 turns this off for
 *                    later calls. Returns the previous setting.
 * rmsq_set_wait_timeout_ns  bound of every device-side wait (default 2e9 ns).
 * rmsq_selftest_wait_timeout  launches one CTA that waits on a barrier nothing will complete,
 *                    bounded by timeout_ns, so a test can check that the bound fires and is
 *                    reported by rmsq_device_status without hanging the GPU.
 * rmsq_debug_convert converts n fp32 values on the device with the kernels' own instructions:
 *                    fmt 0 = E4M3 (one code per byte), 1 = E2M1 (one code per byte, low nibble).
 *                    in and out are device pointers.
 * ------------------------------------------------------------------------------------------- */
int rmsq_set_schedule(int schedule);
rmsq_status rmsq_set_tuning(int stages, int ctas_per_sm, int vectors_per_thread);
rmsq_status rmsq_set_row_warps(int warps_per_cta);
rmsq_status rmsq_set_cluster_size(int ctas_per_cluster);
int rmsq_set_dynamic_rows(int enable);
int rmsq_set_pdl(int enable);
void rmsq_set_wait_timeout_ns(uint64_t timeout_ns);
rmsq_status rmsq_selftest_wait_timeout(uint64_t timeout_ns, void* stream);
rmsq_status rmsq_debug_convert(int fmt, const float* in, uint8_t* out, int64_t n, void* stream);

/* Kernel launches issued by this library in this process (for launch accounting). */
uint64_t rmsq_launch_count(void);

/* ---------------------------------------------------------------------------------------------
 * rmsq_plan -- the launch plan an entry point would choose now for rows of `hidden` elements:
 * schedule, vectors per thread, CTA size, ring depth, cluster size and shared memory, tuning
 * settings included (the same planner the entry points call). A diagnostic; it launches nothing.
 *
 *   mode           0 = rmsnorm_quant_fp8, 1 = rmsnorm_quant_nvfp4, 2 = rmsnorm_quant_mxfp4,
 *                  3 = rmsnorm_nvfp4_global_scale
 *   dtype, residual (0 or 1), weight_offset, hidden   as in the entry points
 *   smem_optin, smem_per_sm, smem_reserved   the device's shared-memory limits in bytes: the
 *                  opt-in maximum per CTA, the total per SM and the part reserved per CTA
 *                  (cudaDevAttrMaxSharedMemoryPerBlockOptin, ...PerMultiprocessor,
 *                  cudaDevAttrReservedSharedMemoryPerBlock; GB300: 232448, 233472, 1024), so the
 *                  plan can be computed without a GPU; smem_optin = 0 takes the current device's
 *   out            receives the plan (caller-owned host memory)
 *
 * Returns RMSQ_ERR_NULL for a NULL out; RMSQ_ERR_DTYPE or RMSQ_ERR_SHAPE as the entry point would
 * for this dtype and width (RMSQ_ERR_SHAPE also for a tuning setting that no plan can honour);
 * RMSQ_ERR_VALUE for an unknown mode, a weight_offset that is not finite or inconsistent limits;
 * RMSQ_ERR_DEVICE when smem_optin = 0 and there is no usable device. The grid (resident CTAs or
 * clusters) is sized at launch from the occupancy API and is not part of the plan.
 * ------------------------------------------------------------------------------------------- */
typedef struct {
    int schedule;            /* 1 CTA per row (bulk-copy ring), 2 register rows, 3 row per warp,
                                4 cluster per row (the values of rmsq_set_schedule) */
    int vectors_per_thread;  /* 16-byte vectors per thread of each row (cluster: of each slice) */
    int threads;             /* threads per CTA */
    int stages;              /* ring slots per CTA (row per warp: per warp; 0 for schedule 2) */
    int cluster;             /* CTAs per cluster (1 unless schedule 4) */
    int smem_bytes;          /* dynamic shared memory per CTA */
    int ctas_per_sm;         /* cap on resident CTAs per SM (0: the occupancy limit) */
    int w16;                 /* 1: 16-bit input with weight_offset 0 (exact packed products) */
} rmsq_plan_info;

rmsq_status rmsq_plan(int mode, int dtype, int residual, float weight_offset, int64_t hidden,
                      int smem_optin, int smem_per_sm, int smem_reserved, rmsq_plan_info* out);

#ifdef __cplusplus
}
#endif

#endif /* RMSQ_H */
