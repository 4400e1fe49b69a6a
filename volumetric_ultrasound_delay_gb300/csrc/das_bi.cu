// BI: batch-inner warp tiling (ffdas paper, Methods, batch-inner paragraphs
// and Algorithm 2; ffdas docs, ALG2).  The record is first permuted to
// K x Q x M x B so that b is contiguous.  A warp owns NW = 32 / G neighbouring
// voxels; the G lanes of a group share one voxel and split its frames: lane t
// holds the 16-byte chunks t, t + G, t + 2G, ... of b, so at every (k, q, m)
// the group reads G consecutive 16-byte vectors (full 32-byte sectors).
//
// Geometry is spread over the group and shared by warp shuffles: for each
// transmit q and each block of G receivers, lane t works out the row, the two
// interpolation weights (and, for IQ, the phase-rotated complex weights) of
// receiver m0 + t, then the group walks the G receivers, broadcasting each
// receiver's values from its lane.
#include "das_device.cuh"

namespace das {
namespace {

constexpr int THREADS = 64;     // 2 warps: 5 % faster than 256 on the 32 x 32-array volume

template <int G, int J, bool CPLX>
__global__ void __launch_bounds__(THREADS)
das_bi_kernel(DasGeom g, const RxPos *__restrict__ rx, const float *__restrict__ perm,
              const float *__restrict__ tau, const float *__restrict__ wtx, float *__restrict__ out)
{
    constexpr int NW = 32 / G;                    // voxels per warp
    constexpr int CH = CPLX ? 2 : 4;              // elements per 16-byte chunk
    using T = typename std::conditional<CPLX, float2, float>::type;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int grp = lane / G;
    const int t = lane % G;
    const int s = (blockIdx.x * (THREADS / 32) + warp) * NW + grp;   // voxel slot
    const bool nvalid = s < g.N;
    const float3 p = nvalid ? voxel_position(g, s) : make_float3(0.f, 0.f, 0.f);
    const int n = nvalid ? voxel_index(g, s) : 0;
    const long long qmb = (long long)g.Q * g.M * g.B;        // row stride of k
    const T *permT = reinterpret_cast<const T *>(perm);

    T acc[J][CH];
#pragma unroll
    for (int c = 0; c < J; ++c)
#pragma unroll
        for (int e = 0; e < CH; ++e) acc[c][e] = T{};

    for (int q = 0; q < g.Q; ++q) {
        const float wq = nvalid ? __ldg(wtx + (long long)q * g.N + n) : 0.f;
        const float tq = nvalid ? fmaf(__ldg(tau + (long long)q * g.N + n), g.fs, -g.t0fs) : 0.f;
        for (int m0 = 0; m0 < g.M; m0 += G) {
            // ---- this lane's receiver m0 + t
            const int m = m0 + t;
            int r0 = 0;
            float w0 = 0.f, w1 = 0.f;
            float2 ph = make_float2(1.f, 0.f);
            if (nvalid && m < g.M) {
                float d;
                if (receive_geometry(g, p, __ldg(rx + m), d)) {
                    const float f = tq + d;
                    if (sample_pair(f, wq, g.K, r0, w0, w1) && CPLX) ph = demod_phase(g, f);
                }
            }
            const int mcount = min(G, g.M - m0);     // warp-uniform
            for (int j = 0; j < mcount; ++j) {
                const int rj = __shfl_sync(0xffffffffu, r0, j, G);
                const float a0 = __shfl_sync(0xffffffffu, w0, j, G);
                const float a1 = __shfl_sync(0xffffffffu, w1, j, G);
                float2 pj = make_float2(1.f, 0.f);
                if constexpr (CPLX) {
                    pj.x = __shfl_sync(0xffffffffu, ph.x, j, G);
                    pj.y = __shfl_sync(0xffffffffu, ph.y, j, G);
                }
                if (a0 == 0.f && a1 == 0.f) continue;   // uniform within the group
                const T *p0 = permT + (long long)rj * qmb + ((long long)q * g.M + m0 + j) * g.B;
                const T *p1 = p0 + qmb;
#pragma unroll
                for (int c = 0; c < J; ++c) {
                    const int b = (t + c * G) * CH;
                    if constexpr (CPLX) {
                        const float4 u0 = __ldg(reinterpret_cast<const float4 *>(p0 + b));
                        const float4 u1 = __ldg(reinterpret_cast<const float4 *>(p1 + b));
                        const float2 W0 = make_float2(a0 * pj.x, a0 * pj.y);
                        const float2 W1 = make_float2(a1 * pj.x, a1 * pj.y);
                        cfma(acc[c][0], W0, make_float2(u0.x, u0.y));
                        cfma(acc[c][1], W0, make_float2(u0.z, u0.w));
                        cfma(acc[c][0], W1, make_float2(u1.x, u1.y));
                        cfma(acc[c][1], W1, make_float2(u1.z, u1.w));
                    } else {
                        const float4 u0 = __ldg(reinterpret_cast<const float4 *>(p0 + b));
                        const float4 u1 = __ldg(reinterpret_cast<const float4 *>(p1 + b));
                        acc[c][0] = fmaf(a0, u0.x, fmaf(a1, u1.x, acc[c][0]));
                        acc[c][1] = fmaf(a0, u0.y, fmaf(a1, u1.y, acc[c][1]));
                        acc[c][2] = fmaf(a0, u0.z, fmaf(a1, u1.z, acc[c][2]));
                        acc[c][3] = fmaf(a0, u0.w, fmaf(a1, u1.w, acc[c][3]));
                    }
                }
            }
        }
    }
    if (!nvalid) return;
    T *outT = reinterpret_cast<T *>(out);
#pragma unroll
    for (int c = 0; c < J; ++c)
#pragma unroll
        for (int e = 0; e < CH; ++e) outT[(long long)((t + c * G) * CH + e) * g.N + n] = acc[c][e];
}

template <int G, int J, bool CPLX>
cudaError_t launch_one(const DasGeom &g, const RxPos *rx, const void *perm, const float *tau,
                       const float *w, void *out, cudaStream_t stream)
{
    constexpr int NW = 32 / G;
    const int voxels_per_block = (THREADS / 32) * NW;
    const int grid = (g.N + voxels_per_block - 1) / voxels_per_block;
    das_bi_kernel<G, J, CPLX><<<grid, THREADS, 0, stream>>>(
        g, rx, static_cast<const float *>(perm), tau, w, static_cast<float *>(out));
    return cudaGetLastError();
}

// lanes per voxel G (default: 16-byte chunks per voxel capped at 16, as the
// pages' N_warp = 2 design) and chunks per lane J
bool choose(int B, bool cplx, int group, int &G, int &J)
{
    const int ch = cplx ? 2 : 4;
    if (B % ch != 0) return false;
    const int chunks = B / ch;
    G = group > 0 ? group : (chunks < 16 ? chunks : 16);
    if (G != 2 && G != 4 && G != 8 && G != 16 && G != 32) return false;
    if (chunks % G != 0) return false;
    J = chunks / G;
    return J == 1 || J == 2 || J == 4;
}

}  // namespace

bool bi_supported(int B, bool cplx, int group)
{
    int G, J;
    return choose(B, cplx, group, G, J);
}

cudaError_t launch_bi(const DasGeom &g, const RxPos *rx, const void *perm, const float *tau,
                      const float *w, void *out, bool cplx, int group, cudaStream_t stream)
{
    int G, J;
    if (!choose(g.B, cplx, group, G, J)) return cudaErrorInvalidValue;
#define DAS_BI_CASE(GG, JJ)                                                                     \
    if (G == GG && J == JJ)                                                                     \
        return cplx ? launch_one<GG, JJ, true>(g, rx, perm, tau, w, out, stream)                \
                    : launch_one<GG, JJ, false>(g, rx, perm, tau, w, out, stream);
    DAS_BI_CASE(2, 1) DAS_BI_CASE(4, 1) DAS_BI_CASE(8, 1) DAS_BI_CASE(16, 1) DAS_BI_CASE(32, 1)
    DAS_BI_CASE(2, 2) DAS_BI_CASE(4, 2) DAS_BI_CASE(8, 2) DAS_BI_CASE(16, 2) DAS_BI_CASE(32, 2)
    DAS_BI_CASE(2, 4) DAS_BI_CASE(4, 4) DAS_BI_CASE(8, 4) DAS_BI_CASE(16, 4) DAS_BI_CASE(32, 4)
#undef DAS_BI_CASE
    return cudaErrorInvalidValue;
}

}  // namespace das
