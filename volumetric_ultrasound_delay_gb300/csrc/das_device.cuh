// Device helpers shared by the DAS kernels: voxel positions, the receive
// geometry, and the rule that turns a fractional sample index into a pair of
// in-record rows with weights.
#pragma once

#include <cuda_runtime.h>

#include <type_traits>

#include "das_internal.cuh"

namespace das {

// Voxel list plans keep the list in a spatially compact order: slot s holds
// the voxel the caller lists at index order[s] (tau_tx, w_tx and y use that
// index).  Grid plans: slot = index.
__device__ __forceinline__ int voxel_index(const DasGeom &g, int s)
{
    return g.order ? __ldg(g.order + s) : s;
}

// position of the voxel in slot n (grid plans: voxel n), sample units
__device__ __forceinline__ float3 voxel_position(const DasGeom &g, int n)
{
    if (g.vox) {
        const float4 p = __ldg(g.vox + n);
        return make_float3(p.x, p.y, p.z);
    }
    const int ix = n % g.nx;
    const int r = n / g.nx;
    const int iy = r % g.ny;
    const int iz = r / g.ny;
    return make_float3(fmaf((float)ix, g.dx, g.x0), fmaf((float)iy, g.dy, g.y0),
                       fmaf((float)iz, g.dz, g.z0));
}

__device__ __forceinline__ float3 voxel_position(const DasGeom &g, int ix, int iy, int iz)
{
    return make_float3(fmaf((float)ix, g.dx, g.x0), fmaf((float)iy, g.dy, g.y0),
                       fmaf((float)iz, g.dz, g.z0));
}

// Receive delay in samples |x - r| and the F-number aperture test
// (2 F#)^2 (dx^2 + dy^2) <= dz^2 with dz > 0 (boundary included).
__device__ __forceinline__ bool receive_geometry(const DasGeom &g, float3 p, RxPos r, float &d)
{
    const float ex = p.x - r.x, ey = p.y - r.y, ez = p.z - r.z;
    const float rho2 = fmaf(ex, ex, ey * ey);
    d = sqrtf(fmaf(ez, ez, rho2));
    return !g.aperture || (ez > 0.f && g.ap2 * rho2 <= ez * ez);
}

// Linear interpolation at fractional index f with weight w, expressed as two
// adjacent in-record rows r0, r0 + 1 (0 <= r0 <= K - 2, so needs K >= 2) and
// their weights.  A sample outside [0, K-1] counts as zero on its own:
//   k0 in [0, K-2]: rows (k0, k0+1), weights (w(1-a), w a)
//   k0 = -1       : only s[0] remains, weight w a   -> rows (0, 1),     (w a, -0)
//   k0 = K-1      : only s[K-1] remains, w(1-a)     -> rows (K-2, K-1), (-0, w(1-a))
//   otherwise (incl. NaN / inf): both weights 0.
// The weight of a row that stands in for a sample outside the record is -0
// (see skip_row): the caller must not read that row, so a non-finite sample
// there cannot reach the sum through a zero weight, while a row inside the
// record is read even when its weight is +0 (a = 0), as the sum's definition
// multiplies it (the other two weights are never -0, even for w = -0).
// Returns false when no sample of the pair lies inside the record.
__device__ __forceinline__ bool sample_pair(float f, float w, int K, int &r0, float &w0, float &w1)
{
    const float fl = floorf(f);
    const bool ok = (fl >= -1.f) && (fl <= (float)(K - 1));
    const float a = f - fl;
    const float u1 = __fadd_rn(w * a, 0.f);      // -0 + 0 = +0
    const float u0 = __fadd_rn(w - u1, 0.f);
    const int k0 = ok ? (int)fl : 0;
    if (!ok) {
        r0 = 0; w0 = 0.f; w1 = 0.f;
    } else if (k0 == -1) {
        r0 = 0; w0 = u1; w1 = -0.f;
    } else if (k0 == K - 1) {
        r0 = K - 2; w0 = -0.f; w1 = u0;
    } else {
        r0 = k0; w0 = u0; w1 = u1;
    }
    return ok;
}

// true for the -0 weight sample_pair gives a row outside the record
__device__ __forceinline__ bool skip_row(float w) { return __float_as_uint(w) == 0x80000000u; }

// exp(+i 2 pi f_demod tau) with tau * fs = f + t0 * fs; the cycle count is
// reduced to [-1/2, 1/2] before the sine/cosine.
__device__ __forceinline__ float2 demod_phase(const DasGeom &g, float f)
{
    float cyc = (f + g.t0fs) * g.fd_over_fs;
    cyc -= rintf(cyc);
    float s, c;
    sincospif(2.f * cyc, &s, &c);
    return make_float2(c, s);
}

// acc += w * s for complex w, s (4 FMA)
__device__ __forceinline__ void cfma(float2 &acc, float2 w, float2 s)
{
    acc.x = fmaf(w.x, s.x, acc.x);
    acc.x = fmaf(-w.y, s.y, acc.x);
    acc.y = fmaf(w.x, s.y, acc.y);
    acc.y = fmaf(w.y, s.x, acc.y);
}

}  // namespace das
