// Internal definitions shared by the libdas CUDA sources (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "das.h"

// Geometry and sizes handed to every DAS kernel by value.  Positions are kept
// in sample units (metres * fs / c), so |x_n - r_m| is directly the receive
// delay in samples and the fractional index is f = tau_tx * fs - t0 * fs + d.
struct DasGeom {
    int nx, ny, nz;
    int N;                // nx * ny * nz, or the length of the voxel list
    float x0, y0, z0;     // first voxel, sample units
    float dx, dy, dz;     // grid spacing, sample units
    float fs;             // Hz, converts tau_tx (s) to samples
    float t0fs;           // t0 * fs
    float ap2;            // (2 F#)^2
    int aperture;         // 0: F# <= 0, every receiver counts
    float fd_over_fs;     // demodulation cycles per sample (IQ)
    int rotate;           // 1: apply the IQ phase
    int B, Q, M, K;
    const float4 *vox;    // voxel list (sample units) in slot order, or nullptr for the grid
    const int *order;     // list plans: caller's index of the voxel in each slot
};

// Receiver record of the plan: position in sample units.
using RxPos = float4;

// Double-precision geometry for float64 / complex128 plans (BL kernel only).
struct Pos64 {
    double x, y, z, pad;
};
struct DasGeom64 {
    int nx, ny, nz;
    int N;
    double x0, y0, z0;    // first voxel, sample units
    double dx, dy, dz;    // grid spacing, sample units
    double fs, t0fs, ap2, fd_over_fs;
    int aperture;
    int B, Q, M, K;
    const Pos64 *vox;     // voxel list (sample units) in slot order, or nullptr for the grid
    const int *order;     // list plans: caller's index of the voxel in each slot
};

namespace das {

// Sets the text das_last_error_string() returns on this thread.
void record_error(const char *msg);

// Launchers (each returns the cudaError_t of its launch).
// Permutes the planes of transmits [q0, q1) (q1 < 0: all Q); to_half converts
// float32 / complex64 elements to half / half2 on the way; nonfinite (device,
// optional) is set to 1 when a permuted float32 value is NaN or inf.
cudaError_t launch_permute(const void *in, void *out, int elem_bytes, int B, int Q, int M, int K,
                           int layout, int num_sms, cudaStream_t stream, int q0 = 0, int q1 = -1,
                           bool to_half = false, unsigned *nonfinite = nullptr);
cudaError_t launch_bl(const DasGeom &g, const RxPos *rx, const void *rf, const float *tau,
                      const float *w, void *out, bool cplx, cudaStream_t stream);
cudaError_t launch_bl64(const DasGeom64 &g, const Pos64 *rx, const void *rf, const float *tau,
                        const float *w, void *out, bool cplx, cudaStream_t stream);
// half: perm holds half / half2 samples (K x Q x M x B)
bool bi_supported(int B, bool cplx, int group, int Q, int M, int K, bool half = false);
cudaError_t launch_bi(const DasGeom &g, const RxPos *rx, const void *perm, const float *tau,
                      const float *w, void *out, bool cplx, int group, cudaStream_t stream,
                      bool half = false);
bool brick_supported(int B, bool cplx, int K, bool half = false);
// Sums transmits [q0, q1) (q1 < 0: all Q) and receivers [m0, m1) (m1 < 0: all
// M; m0 a multiple of 32); with accumulate, adds to out instead of overwriting
// it; half: perm holds half / half2 samples.
cudaError_t launch_brick(const DasGeom &g, const RxPos *rx, const void *perm, const float *tau,
                         const float *w, void *out, bool cplx, cudaStream_t stream, int q0 = 0,
                         int q1 = -1, bool accumulate = false, bool half = false, int m0 = 0,
                         int m1 = -1);
bool pair_supported(int B, bool cplx, int K, bool half = false);
size_t pair_smem_bytes(int B, int Q);
// float32 records; nonfinite: the flag the permute of this record set (the
// kernel then adds each term to its own voxel only); transmits [q0, q1),
// accumulate as for the brick kernel
cudaError_t launch_pair(const DasGeom &g, const RxPos *rx, const void *perm, const float *tau,
                        const float *w, void *out, const unsigned *nonfinite, cudaStream_t stream,
                        int q0 = 0, int q1 = -1, bool accumulate = false);
bool window_supported(int B, bool cplx, int K, int Q, int M, bool half = false);
// float32 records only; transmits [q0, q1), accumulate as for the brick kernel
cudaError_t launch_window(const DasGeom &g, const RxPos *rx, const void *perm, const float *tau,
                          const float *w, void *out, cudaStream_t stream, int q0 = 0, int q1 = -1,
                          bool accumulate = false);

}  // namespace das
