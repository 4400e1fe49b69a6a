// BI: batch-inner warp tiling (ffdas paper, Methods, batch-inner paragraphs
// and Algorithm 2; ffdas docs, ALG2).  The record is first permuted to
// K x Q x M x B so that b is contiguous, here with a zero plane before k = 0
// and one after k = K - 1 ((K+2) x Q x M x B, sample k at plane k + 1): a
// pair that hangs over either end of the record reads a zero row, so every
// pair reads planes k0 + 1 and k0 + 2 and needs no edge cases.  A warp owns NW = 32 / G neighbouring
// voxels; the G lanes of a group share one voxel and split its frames: lane t
// holds the 16-byte chunks t, t + G, t + 2G, ... of b, so at every (k, q, m)
// the group reads G consecutive 16-byte vectors (full 32-byte sectors).
//
// Geometry is spread over the group and shared by warp shuffles.  The CTA
// first stages its voxels' transmit delays and weights in shared memory.  For
// each block of G receivers, lane t works out the distance of receiver m0 + t
// to the group's voxel and the F-number test once; then, per transmit q, the
// lane turns them into a row and two interpolation weights (IQ: and the
// demodulation phase).  A ballot gives each group the receivers of the block
// that contribute, and the group walks only those, U at a time, broadcasting
// from each receiver's lane the 32-bit index (in 16-byte chunks) of its first
// row and its two weights, and issuing the row loads of the U receivers
// before their FMAs.  Real frames are accumulated in pairs
// with the packed FP32 FMA (__ffma2_rn).
//
// With half-precision storage (the pages' BI-FP16 variant: ffdas paper,
// Methods, FP16 paragraphs; ffdas docs, "Mixed-precision storage") the copy
// holds half (real) or half2 (IQ) samples, a 16-byte chunk carries twice as
// many frames, and each is converted to float32 before the interpolation and
// the accumulation.
#include <cuda_fp16.h>

#include "das_device.cuh"

#ifndef DAS_BI_U
#define DAS_BI_U 2
#endif

namespace das {
namespace {

constexpr int THREADS = 64;     // 2 warps per CTA
// resident CTAs per SM the register allocation must allow: 24 (48 warps, 40
// registers, a few bytes of spill) against 21 at the unconstrained 46
// registers: 32 x 32-array volume 20.1 -> 18.6 ms; 28 or 32 CTAs spill more
// and run 21 ms
constexpr int MIN_BLOCKS = 24;

// receivers per walk step: 2 for real data (32-frame float32 volume: 1 step
// 30.0 ms, 2 21.7 ms, 4 28.9 ms); 1 for IQ, whose rows of 64 complex frames
// leave no registers for a second receiver (65.7 ms against 75.9 ms)
template <bool CPLX>
constexpr int walk_step() { return CPLX ? 1 : DAS_BI_U; }

// elements per 16-byte chunk of the copy
template <bool CPLX, bool HALF>
constexpr int chunk_elems() { return HALF ? (CPLX ? 4 : 8) : (CPLX ? 2 : 4); }

// 16 bytes of samples -> NPC float2 values in float32: frame pairs (real) or
// one complex frame each (IQ)
template <bool HALF, int NPC>
__device__ __forceinline__ void unpack_chunk(uint4 u, float2 (&v)[NPC])
{
    if constexpr (HALF) {
        const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
        for (int i = 0; i < NPC; ++i) v[i] = __half22float2(h[i]);
    } else {
        const float2 *f = reinterpret_cast<const float2 *>(&u);
#pragma unroll
        for (int i = 0; i < NPC; ++i) v[i] = f[i];
    }
}

template <int G, int J, bool CPLX, bool HALF>
__global__ void __launch_bounds__(THREADS, MIN_BLOCKS)
das_bi_kernel(DasGeom g, const RxPos *__restrict__ rx, const void *__restrict__ perm,
              const float *__restrict__ tau, const float *__restrict__ wtx, float *__restrict__ out)
{
    constexpr int NW = 32 / G;                    // voxels per warp
    constexpr int CH = chunk_elems<CPLX, HALF>(); // elements per 16-byte chunk
    constexpr int NPC = CPLX ? CH : CH / 2;       // float2 accumulators per chunk
    constexpr int U = walk_step<CPLX>();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int grp = lane / G;
    const int t = lane % G;
    const unsigned gmask = G == 32 ? 0xffffffffu : ((1u << G) - 1u) << (grp * G);  // this group's lanes
    const int s = (blockIdx.x * (THREADS / 32) + warp) * NW + grp;   // voxel slot
    const bool nvalid = s < g.N;
    const float3 p = nvalid ? voxel_position(g, s) : make_float3(0.f, 0.f, 0.f);
    const int n = nvalid ? voxel_index(g, s) : 0;
    const long long qmb = (long long)g.Q * g.M * g.B;        // row stride of k
    const uint4 *perm4 = reinterpret_cast<const uint4 *>(perm) + t;     // chunk t of a row
    const long long qmbc = qmb / CH;                                    // row stride in chunks
    const long long bc = g.B / CH;                                      // chunks per (q, m) row

    // per-voxel transmit delay (samples) and weight, once per CTA
    extern __shared__ float2 txs[];     // [THREADS / 32 * NW][Q]
    for (int e = threadIdx.x; e < (THREADS / 32) * NW * g.Q; e += THREADS) {
        const int v = e / g.Q, q = e % g.Q;
        const int sv = blockIdx.x * (THREADS / 32) * NW + v;
        float2 val = make_float2(0.f, 0.f);
        if (sv < g.N) {
            const int nv = voxel_index(g, sv);
            val = make_float2(fmaf(__ldg(tau + (long long)q * g.N + nv), g.fs, -g.t0fs),
                              __ldg(wtx + (long long)q * g.N + nv));
        }
        txs[e] = val;
    }
    __syncthreads();
    const float2 *txv = txs + (warp * NW + grp) * g.Q;

    // real: frame pairs; IQ: one complex frame each (NPC per chunk)
    float2 acc[J][NPC];
#pragma unroll
    for (int c = 0; c < J; ++c)
#pragma unroll
        for (int i = 0; i < NPC; ++i) acc[c][i] = make_float2(0.f, 0.f);

    for (int m0 = 0; m0 < g.M; m0 += G) {
        // ---- this lane's receiver m0 + t: distance and aperture, for every q
        const int m = m0 + t;
        float d = 0.f;
        const bool ap = nvalid && m < g.M && receive_geometry(g, p, __ldg(rx + m), d);
        if (__ballot_sync(0xffffffffu, ap) == 0u) continue;   // no voxel of the warp sees the block
        for (int q = 0; q < g.Q; ++q) {
            int r0 = 0;
            float w0 = 0.f, w1 = 0.f;
            float2 ph = make_float2(1.f, 0.f);
            bool ok = false;
            if (ap) {
                const float2 tw = txv[q];
                const float f = tw.x + d;
                const float fl = floorf(f);
                // a sample inside the record; false for NaN / inf
                ok = fl >= -1.f && fl <= (float)(g.K - 1);
                if (ok) {
                    r0 = (int)fl + 1;                 // padded plane of sample k0
                    w1 = tw.y * (f - fl);
                    w0 = tw.y - w1;
                    if (CPLX) ph = demod_phase(g, f);
                }
            }
            // chunk index of the first row of this lane's pair
            const unsigned cidx = ok ? (unsigned)((long long)r0 * qmbc + ((long long)q * g.M + m) * bc) : 0u;
            // the group's contributing receivers of the block (same for all its lanes)
            unsigned mine = __ballot_sync(0xffffffffu, ok) & gmask;
            while (mine) {
                // the next U receivers of the list (the lanes holding their values)
                int src[U];
                bool use[U];
                src[0] = __ffs(mine) - 1;
                use[0] = true;
                mine &= mine - 1u;
#pragma unroll
                for (int u = 1; u < U; ++u) {
                    use[u] = mine != 0u;
                    src[u] = use[u] ? __ffs(mine) - 1 : src[0];
                    mine &= mine - 1u;
                }
                uint4 v0[U][J], v1[U][J];
                float2 W0[U], W1[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const unsigned cj = __shfl_sync(gmask, cidx, src[u]);
                    const float a0 = __shfl_sync(gmask, w0, src[u]);
                    const float a1 = __shfl_sync(gmask, w1, src[u]);
                    float2 pj = make_float2(1.f, 0.f);
                    if constexpr (CPLX) {
                        pj.x = __shfl_sync(gmask, ph.x, src[u]);
                        pj.y = __shfl_sync(gmask, ph.y, src[u]);
                    }
                    W0[u] = CPLX ? make_float2(a0 * pj.x, a0 * pj.y) : make_float2(a0, a0);
                    W1[u] = CPLX ? make_float2(a1 * pj.x, a1 * pj.y) : make_float2(a1, a1);
                    const uint4 *p0 = perm4 + cj;
#pragma unroll
                    for (int c = 0; c < J; ++c) {
                        v0[u][c] = make_uint4(0u, 0u, 0u, 0u);
                        v1[u][c] = v0[u][c];
                        if (use[u]) {
                            v0[u][c] = __ldg(p0 + c * G);
                            v1[u][c] = __ldg(p0 + qmbc + c * G);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (!use[u]) break;
#pragma unroll
                    for (int c = 0; c < J; ++c) {
                        float2 x0[NPC], x1[NPC];
                        unpack_chunk<HALF, NPC>(v0[u][c], x0);
                        unpack_chunk<HALF, NPC>(v1[u][c], x1);
#pragma unroll
                        for (int i = 0; i < NPC; ++i) {
                            if constexpr (CPLX) {
                                cfma(acc[c][i], W1[u], x1[i]);
                                cfma(acc[c][i], W0[u], x0[i]);
                            } else {
                                acc[c][i] = __ffma2_rn(W1[u], x1[i], acc[c][i]);
                                acc[c][i] = __ffma2_rn(W0[u], x0[i], acc[c][i]);
                            }
                        }
                    }
                }
            }
        }
    }
    if (!nvalid) return;
#pragma unroll
    for (int c = 0; c < J; ++c) {
        const long long e0 = (long long)(t + c * G) * CH;     // first element of the lane's chunk
#pragma unroll
        for (int i = 0; i < NPC; ++i) {
            if constexpr (CPLX) {
                reinterpret_cast<float2 *>(out)[(e0 + i) * g.N + n] = acc[c][i];
            } else {
                out[(e0 + 2 * i) * g.N + n] = acc[c][i].x;
                out[(e0 + 2 * i + 1) * g.N + n] = acc[c][i].y;
            }
        }
    }
}

// shared memory of a CTA: the transmit table of its voxels
size_t smem_bytes(int G, int Q) { return sizeof(float2) * (size_t)(THREADS / 32) * (32 / G) * Q; }
constexpr size_t SMEM_MAX = 227 * 1024;

template <int G, int J, bool CPLX, bool HALF>
cudaError_t launch_one(const DasGeom &g, const RxPos *rx, const void *perm, const float *tau,
                       const float *w, void *out, cudaStream_t stream)
{
    constexpr int NW = 32 / G;
    const int voxels_per_block = (THREADS / 32) * NW;
    const int grid = (g.N + voxels_per_block - 1) / voxels_per_block;
    const size_t smem = smem_bytes(G, g.Q);
    if (smem > SMEM_MAX) return cudaErrorInvalidValue;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(das_bi_kernel<G, J, CPLX, HALF>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    das_bi_kernel<G, J, CPLX, HALF><<<grid, THREADS, smem, stream>>>(
        g, rx, perm, tau, w, static_cast<float *>(out));
    return cudaGetLastError();
}

// lanes per voxel G (default: 16-byte chunks per voxel capped at 16, as the
// pages' N_warp = 2 design) and chunks per lane J; half storage takes one
// chunk per lane (J = 1)
bool choose(int B, bool cplx, bool half, int group, int &G, int &J)
{
    const int ch = half ? (cplx ? 4 : 8) : (cplx ? 2 : 4);
    if (B % ch != 0) return false;
    const int chunks = B / ch;
    G = group > 0 ? group : (chunks < 16 ? chunks : 16);
    if (G != 2 && G != 4 && G != 8 && G != 16 && G != 32) return false;
    if (chunks % G != 0) return false;
    J = chunks / G;
    return half ? J == 1 : (J == 1 || J == 2 || J == 4);
}

}  // namespace

bool bi_supported(int B, bool cplx, int group, int Q, int M, int K, bool half)
{
    int G, J;
    // row indices travel as 32-bit counts of 16-byte chunks of the padded copy
    const long long chunks = (long long)(K + 2) * Q * M * B / (half ? (cplx ? 4 : 8) : (cplx ? 2 : 4));
    return choose(B, cplx, half, group, G, J) && smem_bytes(G, Q) <= SMEM_MAX && chunks < (1LL << 32);
}

cudaError_t launch_bi(const DasGeom &g, const RxPos *rx, const void *perm, const float *tau,
                      const float *w, void *out, bool cplx, int group, cudaStream_t stream, bool half)
{
    int G, J;
    if (!bi_supported(g.B, cplx, group, g.Q, g.M, g.K, half) || !choose(g.B, cplx, half, group, G, J))
        return cudaErrorInvalidValue;
#define DAS_BI_CASE(GG, JJ, HH)                                                                 \
    if (G == GG && J == JJ && half == HH)                                                       \
        return cplx ? launch_one<GG, JJ, true, HH>(g, rx, perm, tau, w, out, stream)            \
                    : launch_one<GG, JJ, false, HH>(g, rx, perm, tau, w, out, stream);
    DAS_BI_CASE(2, 1, false) DAS_BI_CASE(4, 1, false) DAS_BI_CASE(8, 1, false)
    DAS_BI_CASE(16, 1, false) DAS_BI_CASE(32, 1, false)
    DAS_BI_CASE(2, 2, false) DAS_BI_CASE(4, 2, false) DAS_BI_CASE(8, 2, false)
    DAS_BI_CASE(16, 2, false) DAS_BI_CASE(32, 2, false)
    DAS_BI_CASE(2, 4, false) DAS_BI_CASE(4, 4, false) DAS_BI_CASE(8, 4, false)
    DAS_BI_CASE(16, 4, false) DAS_BI_CASE(32, 4, false)
    DAS_BI_CASE(2, 1, true) DAS_BI_CASE(4, 1, true) DAS_BI_CASE(8, 1, true)
    DAS_BI_CASE(16, 1, true) DAS_BI_CASE(32, 1, true)
#undef DAS_BI_CASE
    return cudaErrorInvalidValue;
}

}  // namespace das
