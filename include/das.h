/*
 * das.h -- C ABI of libdas, volumetric delay-and-sum (DAS) beamforming on one
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (ffdas paper, "ffdas: volumetric ultrasound reconstruction at
 * warp speed", Methods, the accumulation it numbers Eq. (2); ffdas docs, "How
 * It Works", section "The computational challenge"):
 *
 *   y[b,n] = sum_q sum_m  w_tx[q,n] * w_rx[m,n] * P_qmn * S_bqm(f_qmn)
 *   f_qmn  = (tau_tx[q,n] + |x_n - r_m| / c - t0) * fs
 *   S(f)   = (1 - a) s[k0] + a s[k0+1],  k0 = floor(f), a = f - k0,
 *            with every sample outside [0, K-1] counting as zero
 *   w_rx   = 1 if dz > 0 and 2 F# rho <= dz else 0  (rho: lateral distance,
 *            dz: depth of the voxel below the receiver; F# <= 0: w_rx = 1)
 *   P_qmn  = exp(+i 2 pi f_demod (tau_tx[q,n] + |x_n - r_m| / c)) for complex
 *            (IQ) records, 1 for real records
 *
 * Transmit delays and weights are inputs per (q, n); receive delays and the
 * aperture weight are computed inside the kernels from the geometry, never
 * from a stored delay table (ffdas paper, Methods, first paragraph; ffdas
 * docs, "The computational challenge").
 *
 * Conventions for every call:
 *  - Device pointers are CUDA device (or managed) memory of the current
 *    device, C-contiguous, and 16-byte aligned; host pointers are ordinary
 *    host memory (page-locked memory makes the host entry point faster).
 *  - The caller owns every buffer it passes in; the library never frees them.
 *  - A call validates its arguments on the host first.  A rejected call
 *    returns an error code, launches nothing and leaves outputs untouched.
 *  - Device work is asynchronous on the given stream unless stated
 *    otherwise; the caller synchronises before reading results.
 *  - No kernel traps, asserts or waits without a bound.
 *  - das_last_error_string() describes the last error of the calling thread.
 */
#ifndef DAS_H
#define DAS_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct das_plan_s *das_plan;

typedef enum {
    DAS_OK = 0,
    DAS_ERR_INVALID_ARG = 1,    /* null pointer, bad size, misaligned buffer ... */
    DAS_ERR_UNSUPPORTED = 2,    /* valid request this kernel/dtype cannot serve */
    DAS_ERR_OUT_OF_MEMORY = 3,  /* device or host allocation failed */
    DAS_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
    DAS_ERR_TIMEOUT = 5         /* reserved: a bounded device wait ran out */
} das_status;

/* Sample type of the RF record and of the output. */
typedef enum {
    DAS_F32 = 0,   /* real float32 RF -> real float32 y */
    DAS_C64 = 1,   /* interleaved complex64 IQ -> complex64 y */
    DAS_F64 = 2,   /* real float64 RF -> float64 y, computed in double; BL kernel only
                      (ffdas docs, ALG1 supports float64 and complex128) */
    DAS_C128 = 3,  /* interleaved complex128 IQ -> complex128 y, in double; BL only */
    DAS_F16 = 4,   /* real half-precision RF -> float32 y: the record as FP16 storage
                      holds it (ffdas paper, Methods, FP16 paragraphs; ffdas docs,
                      "Mixed-precision storage"), copied bit for bit by the permute and
                      converted to float32 before interpolation; brick and BI kernels */
    DAS_C32H = 5   /* interleaved half2 IQ (real, imaginary half precision) -> complex64
                      y; as DAS_F16 */
} das_dtype;

/* Kernel choice (das_plan_set_option(DAS_OPT_KERNEL, ...)). */
typedef enum {
    DAS_KERNEL_AUTO = 0,   /* brick kernel when it supports the plan, else BI, else BL */
    DAS_KERNEL_BL = 1,     /* per-voxel baseline on the native B x Q x M x K record
                              (ffdas paper, Methods, baseline paragraph / Algorithm 1;
                              ffdas docs, ALG1) */
    DAS_KERNEL_BI = 2,     /* batch-inner warp tiling on a K x Q x M x B copy
                              (ffdas paper, Methods, batch-inner paragraphs /
                              Algorithm 2; ffdas docs, ALG2); the transmit delays
                              and weights of a CTA's voxels sit in shared memory,
                              so Q is limited to 227 KB / (8 B x voxels per CTA),
                              at least 908; rows are indexed in 32 bits of 16-byte
                              chunks, so the record is below 64 GiB */
    DAS_KERNEL_BRICK = 3,  /* this library's sm_103a design: voxel bricks per CTA,
                              per-(voxel, transmit, receiver) geometry staged in
                              shared memory, receivers outside every aperture of
                              the brick skipped, zero-padded Q x M x (K+3) x B copy */
    DAS_KERNEL_WINDOW = 4, /* this library's second sm_103a design on the same copy:
                              a group of lanes owns a 2 x 2 quad of voxels and loads
                              the window of rows the quad needs for a (transmit,
                              receiver) once, with one coefficient per voxel and row.
                              float32 records with B in {8, 16, 32} only; a non-finite
                              sample reaches every voxel of a quad whose window holds its
                              row (zero weight times inf/NaN); on request
                              (AUTO keeps the brick kernel, faster on the workloads
                              measured so far) */
    DAS_KERNEL_PAIR = 5    /* this library's third sm_103a design on the same copy: a
                              group of lanes owns two neighbouring voxels and, per
                              (transmit, receiver), loads the two or three rows their
                              sample pairs span once, applying both voxels' weights to
                              them; float32 records with B in {16, 32, 64}; exact for
                              non-finite samples too (the permute flags them and the
                              kernel then adds every term to its own voxel only) */
} das_kernel;

/* Plan options. */
typedef enum {
    DAS_OPT_KERNEL = 0,    /* das_kernel value */
    DAS_OPT_DEMOD_HZ = 1,  /* f_demod in Hz for DAS_C64 plans (default 0: no rotation);
                              non-zero on a DAS_F32 plan is DAS_ERR_UNSUPPORTED */
    DAS_OPT_TIMING = 2,    /* 1: record CUDA events around the permute and the DAS
                              kernel of each das_beamform (read them with
                              das_plan_last_times); 0 (default): no events */
    DAS_OPT_BI_GROUP = 3,  /* BI kernel: lanes per voxel G in {2,4,8,16,32}; 0 = automatic */
    DAS_OPT_STORAGE = 5,   /* das_storage value: element type of the permuted copy */
    DAS_OPT_RX_GROUPS = 6, /* das_beamform with the brick kernel: number of launches the
                              receivers are split into (contiguous blocks of 32 receivers;
                              each launch adds its receivers' terms to y), so the CTAs
                              resident at one time read a 1/R share of the record; 1
                              (default) = one launch, 0 = enough launches for one share to
                              fit in half the L2.  Changes the float32 summation order,
                              not the result beyond it */
    DAS_OPT_TX_GROUPS = 7, /* das_beamform with the brick kernel: number of launches the
                              transmits are split into (contiguous ranges of transmits;
                              each launch adds its transmits' terms to y), so the CTAs
                              resident at one time read rows of fewer slabs and the rows
                              they share stay in L2; 0 (default) = automatic: one launch
                              when the permuted record holds less than one byte per 64
                              accumulations (B*N*Q*M), else enough launches for one
                              group's share of it to be at most 16 times the L2 size (2
                              for 32 frames x 9 transmits x 1024 receivers x 2048 float32
                              samples and 64^3 voxels on a 126 MB L2); 1 = one launch; at
                              most Q launches are made.  Combines with
                              DAS_OPT_RX_GROUPS (R x T launches).  Changes the float32
                              summation order, not the result beyond it */
    DAS_OPT_HOST_GROUPS = 4 /* das_beamform_host with the brick or window kernel: number of transmit
                              groups the record is streamed in (copy of group g+1
                              overlapping the permute and sum of group g); 0 (default) =
                              min(Q, 5), 1 = copy everything first.  Summing in groups
                              changes the float32 rounding order, not the result beyond it */
} das_option;

/* Element type of the permuted copy of the record (DAS_OPT_STORAGE).
 * DAS_STORAGE_F16 rounds each float32 sample (complex64: each component) to
 * half precision in the permute and converts back to float32 before the
 * interpolation and the sum (ffdas paper, Methods, FP16 paragraphs; ffdas docs,
 * "Mixed-precision storage"): it halves the bytes the kernel reads, and y is
 * then DAS of the half-rounded record.  Served by the brick kernel (B * 2
 * bytes, complex B * 4, a multiple of 16) and by the BI kernel (the pages'
 * BI-FP16 variant, one 16-byte chunk per lane: B in {16, 32, 64, 128} for
 * real records, {8, 16, 32, 64} for IQ); the other kernels return
 * DAS_ERR_UNSUPPORTED. */
typedef enum {
    DAS_STORAGE_NATIVE = 0,
    DAS_STORAGE_F16 = 1
} das_storage;

/* Regular voxel grid: voxel n = ix + nx*(iy + ny*iz) sits at
 * (x0 + ix*dx, y0 + iy*dy, z0 + iz*dz), metres.  The receivers face +z.
 * xyz (optional, may be NULL): host N x 3 float32 positions (metres) of the
 * N = nx*ny*nz voxels in the order n; when given, das_plan_create builds a
 * voxel-list plan (as das_plan_create_points) and origin and spacing are
 * ignored. */
typedef struct {
    int nx, ny, nz;
    float x0, y0, z0;
    float dx, dy, dz;
    const float *xyz;
} das_grid;

/*
 * Creates a plan for fixed geometry and sizes (ffdas paper, Methods: geometry
 * on the fly; the call follows the problem statement of the method).
 *   grid     host, regular voxel grid (N = nx*ny*nz voxels), copied; with
 *            grid->xyz set, the explicit voxel list of das_plan_create_points.
 *   rx_xyz   host, M x 3 float32 receiver positions (metres), copied.
 *   c, fs    speed of sound (m/s) and sampling rate (Hz), both > 0.
 *   t0       time of sample 0 (seconds).
 *   fnum     receive F-number; <= 0 disables the aperture.
 *   dtype    DAS_F32, DAS_C64, DAS_F64 or DAS_C128 (these two: BL kernel,
 *            double-precision geometry and arithmetic; tau_tx and w_tx stay
 *            float32), DAS_F16 or DAS_C32H (brick and BI kernels; a record
 *            already in half precision: half the bytes to copy and permute,
 *            the same arithmetic as DAS_OPT_STORAGE = DAS_STORAGE_F16, which
 *            is implied and may be set either way).
 *   B,Q,M,K  frames, transmits, receivers, samples per record (all >= 1);
 *            Q*M*(K+3) and B*N must stay below 2^31, K below 2^22.
 * Allocates the device copies of the geometry; the permute scratch of the BI,
 * brick and window kernels (B*Q*M*(K+3) elements) is allocated on first use.
 * A plan's device memory comes from CUDA's stream-ordered allocator (the
 * device's default memory pool) on a stream the plan owns.
 * Errors: DAS_ERR_INVALID_ARG, DAS_ERR_OUT_OF_MEMORY, DAS_ERR_CUDA; *plan is
 * set to NULL on failure.  The plan belongs to the device current at creation.
 */
das_status das_plan_create(das_plan *plan, const das_grid *grid, const float *rx_xyz,
                           float c, float fs, float t0, float fnum, das_dtype dtype,
                           int B, int Q, int M, int K);

/*
 * Plan over an explicit list of voxel positions instead of a regular grid: the
 * sparse-voxel form of the operation (ffdas docs, "How It Works", das_sparse
 * in "Mixed-precision storage" and "Other operations").  y and the Q x N
 * tau_tx / w_tx arrays are indexed by list position n.
 *   voxel_xyz  host, N x 3 float32 positions (metres), copied.
 *   other arguments as das_plan_create.
 * The plan keeps the list in its own spatially compact order (depth bands,
 * deepest first, then a Morton curve in x-y on cells of the list's mean
 * spacing), so the bricks of the brick and window kernels are neighbours in
 * space whatever order the caller lists the voxels in; y, tau_tx and w_tx
 * stay in the caller's order.
 * Errors: as das_plan_create.
 */
das_status das_plan_create_points(das_plan *plan, const float *voxel_xyz, int N,
                                  const float *rx_xyz, float c, float fs, float t0, float fnum,
                                  das_dtype dtype, int B, int Q, int M, int K);

/* Sets / reads one das_option.  No passage of the pages defines this call: it
 * is library plumbing that selects among the pages' kernels (BL, BI) and this
 * library's own, and carries the IQ demodulation frequency of the IQ form of
 * the sum (ffdas docs, "How It Works", "Mixed-precision storage": complex
 * records) and the FP16 storage switch (ffdas paper, Methods, FP16
 * paragraphs).  Takes effect from the next das_beamform; host only, no device
 * work.  Errors: DAS_ERR_INVALID_ARG (null plan, unknown option or value),
 * DAS_ERR_UNSUPPORTED (see DAS_OPT_DEMOD_HZ). */
das_status das_plan_set_option(das_plan plan, int option, double value);
das_status das_plan_get_option(das_plan plan, int option, double *value);

/* The kernel das_beamform will run for this plan (after AUTO resolution). */
das_status das_plan_kernel(das_plan plan, int *kernel);

/* Kernel launches one das_beamform makes with the plan's current options: the
 * permute (none for BL) plus the DAS launches (DAS_OPT_RX_GROUPS x
 * DAS_OPT_TX_GROUPS for the brick kernel, else one).  No passage of the pages
 * defines this call: it is library plumbing for profiling and accounting.
 * Host only.  Errors: DAS_ERR_INVALID_ARG (NULL argument). */
das_status das_plan_launches(das_plan plan, int *launches);

/*
 * y = DAS(rf) on the device (the formula at the top of this file).
 *   rf       device, B x Q x M x K, k contiguous, of the plan's dtype (float32,
 *            interleaved complex64, float64, complex128, float16 or interleaved
 *            half2).
 *   tau_tx   device, Q x N float32 transmit delays (seconds).
 *   w_tx     device, Q x N float32 transmit weights.
 *   out      device, B x N: float32 (DAS_F32, DAS_F16), complex64 (DAS_C64,
 *            DAS_C32H), float64 or complex128; fully overwritten.
 *   stream   CUDA stream of the plan's device (0 = legacy default stream).
 * The BI, brick and window kernels first permute rf into the plan's scratch (ffdas
 * paper, Methods, batch-inner paragraph; ffdas docs, ALG2: permuted as part of
 * the launch), so one plan must not run two das_beamform calls at once; use one
 * plan per concurrent stream.
 * The brick kernel on float32 records scales each transmit weight by at most
 * 2^9 (an exact power of two) before forming the interpolation weights, so
 * weights of magnitude above 2^119 (about 6.6e35) overflow there; every
 * smaller weight gives the same float32 products as the unscaled arithmetic.
 * Errors: DAS_ERR_INVALID_ARG (null or misaligned pointers), DAS_ERR_UNSUPPORTED
 * (kernel cannot serve this plan), DAS_ERR_OUT_OF_MEMORY (scratch), DAS_ERR_CUDA
 * (launch failure).  Asynchronous.
 */
das_status das_beamform(das_plan plan, const void *rf, const float *tau_tx,
                        const float *w_tx, void *out, cudaStream_t stream);

/*
 * The same computation from host buffers (same layouts as das_beamform, host
 * memory): copies the inputs to plan-owned device buffers, computes, copies y
 * back and synchronises `stream` before returning.  With the brick or window kernel the
 * record is streamed in groups of transmits (DAS_OPT_HOST_GROUPS) on an internal
 * copy stream, so the copy of one group overlaps the permute and sum of the
 * previous one; the other kernels copy everything, then run das_beamform.
 * Device buffers (about the size of rf) and the copy stream are created on first
 * use and kept.  Page-locked host memory is needed for the overlap.  Different
 * plans may be driven from different host threads at once (each call blocks
 * only its own thread), which overlaps one volume's upload with another's
 * kernels; one plan serves one call at a time.
 * Errors: as das_beamform.  Synchronous.
 */
das_status das_beamform_host(das_plan plan, const void *rf_host, const float *tau_tx_host,
                             const float *w_tx_host, void *out_host, cudaStream_t stream);

/*
 * A stream of volumes from host buffers: n_volumes records acquired with the
 * same transmits, one after another in rf_host (n_volumes x B x Q x M x K,
 * each in the layout of das_beamform_host), beamformed with the one tau_tx /
 * w_tx (Q x N, host) into out_host (n_volumes x B x N), in order.  The record of
 * volume v + 1 is copied to the device, group of transmits by group, while the
 * kernels of volume v run: a group's copy waits only until volume v's permute
 * has read that group's staging copy, so the host link and the kernels stay
 * busy across volumes (the pages' streaming use, "kilohertz volume rates":
 * ffdas docs, "How It Works").  Same arithmetic and output, bit for bit, as
 * das_beamform_host on each volume.  Page-locked host memory is needed for the
 * overlap.  Device buffers as das_beamform_host.
 * Errors: as das_beamform_host, and DAS_ERR_INVALID_ARG for n_volumes < 1.
 * Synchronous (returns when every y is in out_host).
 */
das_status das_beamform_host_volumes(das_plan plan, int n_volumes, const void *rf_host,
                                     const float *tau_tx_host, const float *w_tx_host, void *out_host,
                                     cudaStream_t stream);

/* Device milliseconds of the permute and of the DAS kernel of the last
 * das_beamform on this plan, when DAS_OPT_TIMING is 1 (synchronises on the
 * recorded events).  permute_ms is 0 for the BL kernel.  Errors:
 * DAS_ERR_INVALID_ARG when timing is off or no call was made yet. */
das_status das_plan_last_times(das_plan plan, float *permute_ms, float *das_ms);

/* Bytes of device memory the plan holds now. */
das_status das_plan_device_bytes(das_plan plan, size_t *bytes);

/* Frees everything the plan owns.  No passage of the pages defines this call:
 * it is library plumbing that ends the life of a plan.
 * It does not wait on the host, neither for this plan's queued work nor for
 * any other stream: the plan's device memory is released in stream order, on
 * the plan's own stream, after the last work that a das_beamform or
 * das_beamform_host of this plan queued on the caller's stream, which still
 * runs to completion and writes its output.  The plan handle is invalid once
 * the call returns.  A NULL plan is a no-op returning DAS_OK. */
das_status das_plan_destroy(das_plan plan);

/*
 * RF layout permute (ffdas paper, Methods, batch-inner paragraph: B x Q x M x K
 * with k contiguous -> a layout with b contiguous).  A bit-exact copy, or with
 * storage DAS_STORAGE_F16 a copy rounded to half precision (round to nearest
 * even; complex: both components), as the half-storage kernels read it.
 *   layout 0: K x Q x M x B (the pages' batch-inner layout, used by BI)
 *   layout 1: Q x M x K x B (rows of one (q, m) adjacent)
 *   layout 2: Q x M x (K+3) x B, sample k of slab (q, m) at row k + 1; rows 0,
 *             K + 1 and K + 2 of every slab are not written (the brick kernel
 *             keeps them zero, so reads just outside the record return 0)
 *   layout 3: (K+2) x Q x M x B, sample k at plane k + 1; planes 0 and K + 1
 *             are not written (the BI kernel keeps them zero)
 *   in       device buffer of B*Q*M*K elements of dtype (DAS_F32, DAS_C64,
 *            DAS_F16 or DAS_C32H; the half types are copied bit for bit, with
 *            either storage value);
 *   out      device buffer of B*Q*M*K (layouts 0, 1), B*Q*M*(K+3) (layout 2) or
 *            B*Q*M*(K+2) (layout 3)
 *            elements of dtype, or of half / half2 with DAS_STORAGE_F16; in and
 *            out must not overlap, and each must be aligned to its element
 *            size (16-byte alignment, with K and B multiples of a 16-byte
 *            vector, selects the vectorised loads and stores).
 * Errors: DAS_ERR_INVALID_ARG, DAS_ERR_CUDA.  Asynchronous.
 */
das_status das_permute(const void *in, void *out, das_dtype dtype, int B, int Q, int M,
                       int K, int layout, das_storage storage, cudaStream_t stream);

/*
 * The batch-inner permute by itself: B x Q x M x K -> K x Q x M x B, bit for
 * bit (ffdas paper, Methods, batch-inner paragraph; ffdas docs, ALG2, the
 * permute done as part of the launch).  Same as das_permute with layout 0 and
 * DAS_STORAGE_NATIVE: dtype DAS_F32 or DAS_C64, in and out device buffers of
 * B*Q*M*K elements, aligned to the element size, that must not overlap.
 * Errors: DAS_ERR_INVALID_ARG, DAS_ERR_CUDA.  Asynchronous.
 */
das_status das_permute_bqmk_to_kqmb(const void *in, void *out, das_dtype dtype, int B, int Q,
                                    int M, int K, cudaStream_t stream);

/*
 * das_beamform_noalloc -- the same computation as a plan running the brick
 * kernel, for callers that cannot allocate device memory.  The ffdas pages
 * have no counterpart to this entry point.
 *
 * Who it is for: code that must not call cudaMalloc once it is running, such as
 * the real-time reconstruction loop of a scanner (cudaMalloc can synchronise the
 * device and stall acquisition) or a host framework that hands out all device
 * memory from its own pool at start-up and forbids other allocations.  A plan
 * allocates, so those callers use this call instead.  It allocates nothing:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 *
 * Arguments are those of das_plan_create and das_beamform together, except that
 *   rx_xyz   is a DEVICE pointer (M x 3 float32 receiver positions, metres), and
 *   f_demod  (Hz, DAS_C64 only; 0 = no rotation) is passed directly, and
 *   dtype    is DAS_F32 or DAS_C64 (other types: DAS_ERR_INVALID_ARG).
 * rf, tau_tx, w_tx and out are device buffers in the layouts of das_beamform.
 *
 * Scratch: one file-scope static device array of 64 MiB (67,108,864 bytes)
 * inside libdas, which every GPU that loads the library's kernels holds until
 * the process exits.  A call needs 16*M (rounded up to 256) +
 * B*Q*M*(K+3)*element-size bytes of it; larger requests are rejected with
 * DAS_ERR_INVALID_ARG and a message naming both sizes, and launch nothing.
 * Every call shares that one array and leaves its contents behind; the call
 * itself clears the part that must start at zero.  Calls whose device work
 * overlaps (unordered streams, or several host threads) race on the array and
 * give wrong results, so serialise them.
 *
 * Each call looks up the array's device address on the current device
 * (cudaGetSymbolAddress, which allocates nothing), so a cudaDeviceReset or
 * another context of the device between calls is harmless.  The first call on
 * each device also loads libdas's kernels there; make that first call before
 * any stream capture.
 *
 * rx_xyz is device memory, so its values are not checked on the host: a
 * non-finite receiver position gives non-finite output rather than an error.
 *
 * Errors: DAS_ERR_INVALID_ARG (NULL or misaligned pointers, bad sizes, scratch
 * too small), DAS_ERR_UNSUPPORTED (B / K the brick kernel cannot serve,
 * f_demod on real data), DAS_ERR_CUDA.  Asynchronous on `stream`.
 */
das_status das_beamform_noalloc(const das_grid *grid, const float *rx_xyz, float c, float fs,
                                float t0, float fnum, double f_demod, das_dtype dtype,
                                int B, int Q, int M, int K, const void *rf,
                                const float *tau_tx, const float *w_tx, void *out,
                                cudaStream_t stream);

/* Text of the last error raised on the calling thread ("" if none): a
 * thread-local buffer owned by the library, valid until the thread's next libdas
 * call.  No passage of the pages defines this call: it is library plumbing. */
const char *das_last_error_string(void);

/* Library version, e.g. "1.0.0". */
const char *das_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DAS_H */
