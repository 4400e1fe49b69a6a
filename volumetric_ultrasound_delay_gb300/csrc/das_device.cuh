// Device helpers shared by the DAS kernels: voxel positions, the receive
// geometry, the IQ demodulation phase and the complex FMA.
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
