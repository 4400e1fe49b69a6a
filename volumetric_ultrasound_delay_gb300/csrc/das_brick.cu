// BRICK: this library's DAS kernel for sm_103a (not a design from the pages).
//
// Each CTA (8 warps) owns a brick of V voxels in one x-y slice (8 x 4 for 32
// frames of float32) and all B frames of them.  Neighbouring voxels of a slice
// need nearly the same sample rows of every receiver, so the warps of a CTA
// walking the same (q, m) at the same time hit the same L1 lines; bricks are
// flat in z because one voxel step in depth moves the delay by many samples.
//
// The record is permuted to Q x M x K x B, so the two rows a voxel reads for a
// (q, m) are adjacent 16 * G * J-byte runs.  A group of G lanes owns one voxel;
// lane t loads the 16-byte chunks t, t + G, ... of both rows (G = 8: one full
// 128-byte line per row and instruction).
//
// Geometry is computed once per (voxel, transmit, receiver) instead of once per
// lane, and staged in shared memory:
//   phase A (per block of 32 receivers): distance |x_v - r_m| in samples and the
//            F-number test for all V voxels (warp = voxel, lane = receiver); a
//            CTA-wide bit mask keeps only receivers inside the aperture of at
//            least one voxel of the brick, so whole receiver blocks outside
//            every aperture cost nothing;
//   phase B (per transmit): row index and the two interpolation weights (IQ:
//            phase-rotated complex weights) of every active (voxel, receiver),
//            double-buffered so one barrier per transmit suffices;
//   phase C: every group walks the active receivers, reading its entry with a
//            broadcast shared-memory load and accumulating 2 rows x its chunks.
#include "das_device.cuh"

namespace das {
namespace {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int MC = 32;                 // receivers per block (one per lane in phase A/B)
constexpr float FAR = 1.0e30f;         // distance marking "outside the aperture"

template <int V>
struct BrickShape {
    static constexpr int BX = V >= 128 ? 16 : (V >= 32 ? 8 : 4);
    static constexpr int BY = V / BX;
};

template <bool CPLX>
struct Weights;
template <>
struct Weights<false> { using type = float2; };    // (w0, w1)
template <>
struct Weights<true> { using type = float4; };     // (W0.re, W0.im, W1.re, W1.im)

template <int G, bool CPLX>
size_t smem_bytes(int Q)
{
    constexpr int V = WARPS * (32 / G);
    using W = typename Weights<CPLX>::type;
    return sizeof(W) * 2 * V * MC + sizeof(int) * 2 * V * MC + sizeof(float) * V * MC +
           sizeof(float2) * (size_t)V * Q + sizeof(unsigned) * 2 * WARPS;
}

template <int G, int J, bool CPLX>
__global__ void __launch_bounds__(THREADS, 4)
das_brick_kernel(DasGeom g, const RxPos *__restrict__ rx, const float *__restrict__ perm,
                 const float *__restrict__ tau, const float *__restrict__ wtx,
                 float *__restrict__ out, int bricks_x, int bricks_y)
{
    constexpr int NW = 32 / G;                     // voxels per warp
    constexpr int V = WARPS * NW;                  // voxels per CTA
    constexpr int BX = BrickShape<V>::BX;
    constexpr int CH = CPLX ? 2 : 4;               // elements per 16-byte chunk
    using T = typename std::conditional<CPLX, float2, float>::type;
    using W = typename Weights<CPLX>::type;

    extern __shared__ __align__(16) unsigned char smem_raw[];
    W *wts = reinterpret_cast<W *>(smem_raw);                        // [2][V][MC]
    int *rows = reinterpret_cast<int *>(wts + 2 * V * MC);           // [2][V][MC]
    float *dist = reinterpret_cast<float *>(rows + 2 * V * MC);      // [V][MC]
    float2 *tx = reinterpret_cast<float2 *>(dist + V * MC);          // [V][Q]  (tau*fs - t0*fs, w)
    unsigned *masks = reinterpret_cast<unsigned *>(tx + V * g.Q);    // [2][WARPS]

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int bx = blockIdx.x % bricks_x;
    const int rb = blockIdx.x / bricks_x;
    const int by = rb % bricks_y;
    const int iz = rb / bricks_y;

    // ---- per-voxel transmit delay (samples) and weight, once per CTA
    for (int e = tid; e < V * g.Q; e += THREADS) {
        const int v = e / g.Q, q = e % g.Q;
        const int ix = bx * BX + v % BX, iy = by * (V / BX) + v / BX;
        float2 val = make_float2(0.f, 0.f);
        if (ix < g.nx && iy < g.ny) {
            const long long n = ix + (long long)g.nx * (iy + (long long)g.ny * iz);
            val.x = fmaf(__ldg(tau + (long long)q * g.N + n), g.fs, -g.t0fs);
            val.y = __ldg(wtx + (long long)q * g.N + n);
        }
        tx[e] = val;
    }

    // ---- consumer identity: group grp of this warp owns voxel cv
    const int grp = lane / G;
    const int t = lane % G;
    const int cv = warp * NW + grp;
    const int cix = bx * BX + cv % BX, ciy = by * (V / BX) + cv / BX;
    const bool cvalid = cix < g.nx && ciy < g.ny;
    const T *permT = reinterpret_cast<const T *>(perm);

    T acc[J][CH];
#pragma unroll
    for (int c = 0; c < J; ++c)
#pragma unroll
        for (int e = 0; e < CH; ++e) acc[c][e] = T{};

    __syncthreads();

    int chunk = 0;
    for (int m0 = 0; m0 < g.M; m0 += MC, ++chunk) {
        // ---- phase A: distances and aperture, warp = voxel, lane = receiver
        unsigned any = 0;
        const int m = m0 + lane;
        const RxPos r = m < g.M ? __ldg(rx + m) : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int v = warp; v < V; v += WARPS) {
            const int ix = bx * BX + v % BX, iy = by * (V / BX) + v / BX;
            float d = FAR;
            if (m < g.M && ix < g.nx && iy < g.ny) {
                float dd;
                if (receive_geometry(g, voxel_position(g, ix, iy, iz), r, dd)) {
                    d = dd;
                    any = 1u;
                }
            }
            dist[v * MC + lane] = d;
        }
        const unsigned bal = __ballot_sync(0xffffffffu, any);
        if (lane == 0) masks[(chunk & 1) * WARPS + warp] = bal;
        __syncthreads();
        unsigned mask = 0;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) mask |= masks[(chunk & 1) * WARPS + w];
        if (mask == 0u) continue;                  // CTA-uniform

        for (int q = 0; q < g.Q; ++q) {
            const int buf = q & 1;
            // ---- phase B: row and weights of every active (voxel, receiver)
            if ((mask >> lane) & 1u) {
                const int rowbase = (q * g.M + m0 + lane) * g.K;
                for (int v = warp; v < V; v += WARPS) {
                    const float2 tw = tx[v * g.Q + q];
                    const float f = tw.x + dist[v * MC + lane];
                    int r0;
                    float w0, w1;
                    const bool nz = sample_pair(f, tw.y, g.K, r0, w0, w1);
                    const int idx = (buf * V + v) * MC + lane;
                    rows[idx] = rowbase + r0;
                    if constexpr (CPLX) {
                        const float2 ph = nz ? demod_phase(g, f) : make_float2(1.f, 0.f);
                        wts[idx] = make_float4(w0 * ph.x, w0 * ph.y, w1 * ph.x, w1 * ph.y);
                    } else {
                        wts[idx] = make_float2(w0, w1);
                    }
                }
            }
            __syncthreads();

            // ---- phase C: accumulate
            const W *wv = wts + (buf * V + cv) * MC;
            const int *rv = rows + (buf * V + cv) * MC;
            unsigned mm = mask;
            while (mm) {
                const int j = __ffs(mm) - 1;
                mm &= mm - 1u;
                const W ww = wv[j];
                bool zero;
                if constexpr (CPLX) zero = ww.x == 0.f && ww.y == 0.f && ww.z == 0.f && ww.w == 0.f;
                else zero = ww.x == 0.f && ww.y == 0.f;
                if (zero) continue;                // uniform within the group
                const T *p0 = permT + (long long)rv[j] * g.B + t * CH;
                const T *p1 = p0 + g.B;
#pragma unroll
                for (int c = 0; c < J; ++c) {
                    const float4 u0 = __ldg(reinterpret_cast<const float4 *>(p0 + c * G * CH));
                    const float4 u1 = __ldg(reinterpret_cast<const float4 *>(p1 + c * G * CH));
                    if constexpr (CPLX) {
                        const float2 W0 = make_float2(ww.x, ww.y), W1 = make_float2(ww.z, ww.w);
                        cfma(acc[c][0], W0, make_float2(u0.x, u0.y));
                        cfma(acc[c][1], W0, make_float2(u0.z, u0.w));
                        cfma(acc[c][0], W1, make_float2(u1.x, u1.y));
                        cfma(acc[c][1], W1, make_float2(u1.z, u1.w));
                    } else {
                        acc[c][0] = fmaf(ww.x, u0.x, fmaf(ww.y, u1.x, acc[c][0]));
                        acc[c][1] = fmaf(ww.x, u0.y, fmaf(ww.y, u1.y, acc[c][1]));
                        acc[c][2] = fmaf(ww.x, u0.z, fmaf(ww.y, u1.z, acc[c][2]));
                        acc[c][3] = fmaf(ww.x, u0.w, fmaf(ww.y, u1.w, acc[c][3]));
                    }
                }
            }
        }
    }

    if (!cvalid) return;
    const long long n = cix + (long long)g.nx * (ciy + (long long)g.ny * iz);
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
    constexpr int V = WARPS * (32 / G);
    constexpr int BX = BrickShape<V>::BX, BY = V / BX;
    const int bricks_x = (g.nx + BX - 1) / BX;
    const int bricks_y = (g.ny + BY - 1) / BY;
    const long long blocks = (long long)bricks_x * bricks_y * g.nz;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const size_t smem = smem_bytes<G, CPLX>(g.Q);
    cudaError_t err = cudaFuncSetAttribute(das_brick_kernel<G, J, CPLX>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    das_brick_kernel<G, J, CPLX><<<(int)blocks, THREADS, smem, stream>>>(
        g, rx, static_cast<const float *>(perm), tau, w, static_cast<float *>(out), bricks_x, bricks_y);
    return cudaGetLastError();
}

bool choose(int B, bool cplx, int &G, int &J)
{
    const int ch = cplx ? 2 : 4;
    if (B % ch != 0) return false;
    const int chunks = B / ch;
    if (chunks <= 8) {
        G = chunks;
        J = 1;
        return G == 2 || G == 4 || G == 8;
    }
    G = 8;
    J = chunks / 8;
    return chunks % 8 == 0 && (J == 2 || J == 4);
}

}  // namespace

bool brick_supported(int B, bool cplx, int K)
{
    int G, J;
    return K >= 2 && choose(B, cplx, G, J);
}

cudaError_t launch_brick(const DasGeom &g, const RxPos *rx, const void *perm, const float *tau,
                         const float *w, void *out, bool cplx, cudaStream_t stream)
{
    int G, J;
    if (g.K < 2 || !choose(g.B, cplx, G, J)) return cudaErrorInvalidValue;
#define DAS_BRICK_CASE(GG, JJ)                                                                  \
    if (G == GG && J == JJ)                                                                     \
        return cplx ? launch_one<GG, JJ, true>(g, rx, perm, tau, w, out, stream)                \
                    : launch_one<GG, JJ, false>(g, rx, perm, tau, w, out, stream);
    DAS_BRICK_CASE(2, 1) DAS_BRICK_CASE(4, 1) DAS_BRICK_CASE(8, 1)
    DAS_BRICK_CASE(8, 2) DAS_BRICK_CASE(8, 4)
#undef DAS_BRICK_CASE
    return cudaErrorInvalidValue;
}

}  // namespace das
