// PAIR: this library's third DAS kernel for sm_103a (not a design from the
// pages).  It attacks what binds the brick kernel: every float32 accumulation
// there returns 8 bytes of samples from L1 to registers (two rows of B frames
// per voxel, transmit and receiver), and the L1 data pipe returns 128 bytes
// per SM and clock.  Two voxels one grid step apart in x need rows that are
// mostly the same or one apart: on the 32 x 32-array volume the rows k0 of the
// two are equal for 34 % of their (transmit, receiver) terms, one apart for
// 53 % and further apart for 14 %.  A group of G lanes therefore owns such a
// pair of voxels and, per term, loads the window of rows k, k + 1 (and k + 2
// when the two k0 differ by one) once, then applies both voxels' interpolation
// weights to it in registers: 2.8 rows per pair instead of 4.
//
// Record layout: the brick kernel's zero-padded Q x M x (K+3) x B copy (sample
// k of slab (q, m) at row k + 1; rows 0, K+1, K+2 zero), so a window that hangs
// over either end of the record reads zero rows.  Lane t of a group loads the
// 16-byte chunk t of a row (G = B * 4 / 16 lanes, one 128-byte line per row
// for 32 float32 frames) and keeps four frames of both voxels.
//
// One warp per CTA, NP = 32 / G pairs (2 NP voxels, x-neighbours paired):
//   phase A (per block of 32 receivers, lane = receiver): distances of the
//            warp's voxels in samples and the F-number test, in registers;
//   phase B (per transmit, lane = receiver): per pair, one entry when both
//            voxels contribute and their k0 differ by at most one (the window
//            starts at the smaller k0, each voxel's offset g in [0, 2) holds its
//            position in the window), else one single-voxel entry per voxel that
//            contributes; a warp ballot compacts each pair's entries into a list
//            in the warp's shared memory (double-buffered by transmit parity);
//   phase C: each group walks its pair's list, U entries per trip, the row loads
//            of the next trip issued before the FMAs of the current one.  Each
//            voxel's weights on the window's three rows are (w(1-a), w a, 0) or
//            (0, w(1-a), w a) by its offset; the FMAs are packed FP32
//            (__ffma2_rn, two frames per instruction).
//
// Weights of zero multiply rows a voxel does not use, which is exact only for
// finite samples.  The permute that writes the copy raises a flag when the
// record holds a non-finite sample; the kernel then makes single-voxel entries
// only and adds each to its own voxel, so NaN and inf reach exactly the
// outputs whose sample pairs hold them, as in the sum's definition.
#include "das_device.cuh"

#ifndef DAS_PAIR_U
#define DAS_PAIR_U 1
#endif
#ifndef DAS_PAIR_MIN_WARPS
#define DAS_PAIR_MIN_WARPS 32
#endif
#ifndef DAS_PAIR_MIN_WARPS_J2
#define DAS_PAIR_MIN_WARPS_J2 28
#endif

namespace das {
namespace {

constexpr int MC = 32;                  // receivers per block (one per lane in phases A and B)
constexpr float FAR = 1.0e30f;          // distance marking "outside the aperture"
constexpr int LIST_STRIDE = 2 * MC + 2; // up to two entries per receiver; 16-byte aligned lists

// warp footprint: NP pairs, two voxels each along x; BX voxels across x, the
// rest in y
#ifndef DAS_PAIR_BX
#define DAS_PAIR_BX 4
#endif
template <int G>
struct PairShape {
    static constexpr int NP = 32 / G;
    static constexpr int V = 2 * NP;
    static constexpr int BX = V >= DAS_PAIR_BX ? DAS_PAIR_BX : 2;
    static constexpr int BY = V / BX;
    static_assert(V % BX == 0, "pairs tile the brick");
};

// shared memory of a CTA: the pairs' entry lists, the distances of phase A
// (voxel-major, one per lane) and the voxels' transmit table
template <int G>
size_t smem_bytes(int Q)
{
    using SH = PairShape<G>;
    return sizeof(uint2) * SH::NP * LIST_STRIDE + sizeof(float) * SH::V * MC +
           sizeof(float2) * (size_t)SH::V * Q;
}

// Entry: x = row << 4 | pA << 3 | pB << 2 | dA << 1 | dB, with the window's
// first row relative to the first row of the block of receivers, pX whether
// voxel X takes part, dX its offset's integer part; y holds the two offsets'
// fractions in 15 bits each, rounded to nearest and kept below one step, over
// a set bit 15 (so a byte permute turns each into a float in [1, 2)).
__device__ __forceinline__ unsigned frac15(float f)
{
    return 0x8000u | min(__float2uint_rn(f * 32768.f), 32767u);
}

__device__ __forceinline__ uint2 make_entry(int rel, float gA, float gB, unsigned present)
{
    const unsigned dA = gA >= 1.f, dB = gB >= 1.f;
    const float aA = gA - (float)dA, aB = gB - (float)dB;
    return make_uint2(((unsigned)rel << 4) | present | (dA << 1) | dB, frac15(aA) | (frac15(aB) << 16));
}

// the offsets' fractions back in [0, 1)
__device__ __forceinline__ float2 fractions(unsigned y)
{
    const float a = __int_as_float(__byte_perm(y, 0x3f000000u, 0x7104)) - 1.f;
    const float b = __int_as_float(__byte_perm(y, 0x3f000000u, 0x7324)) - 1.f;
    return make_float2(a, b);
}

// J contiguous 16-byte chunks of a row (one 256-bit load for J = 2)
template <int J>
__device__ __forceinline__ void load_chunks(const char *p, uint4 (&v)[J])
{
    if constexpr (J == 2) {
        asm("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
            : "=r"(v[0].x), "=r"(v[0].y), "=r"(v[0].z), "=r"(v[0].w),
              "=r"(v[1].x), "=r"(v[1].y), "=r"(v[1].z), "=r"(v[1].w)
            : "l"(p));
    } else {
#pragma unroll
        for (int c = 0; c < J; ++c) v[c] = __ldg(reinterpret_cast<const uint4 *>(p) + c);
    }
}

template <int U, int J>
struct PTrip {
    uint2 e[U];
    uint4 s[U][3][J];
};

template <int J>
constexpr int min_blocks() { return J == 1 ? DAS_PAIR_MIN_WARPS : DAS_PAIR_MIN_WARPS_J2; }

template <int G, int J>
__global__ void __launch_bounds__(32, min_blocks<J>())
das_pair_kernel(DasGeom g, const RxPos *__restrict__ rx, const void *__restrict__ perm,
                const float *__restrict__ tau, const float *__restrict__ wtx,
                float *__restrict__ out, int bricks_x, int bricks_y, const unsigned *nonfinite,
                int q_begin, int q_end, int add_to_out)
{
    using SH = PairShape<G>;
    constexpr int NP = SH::NP, V = SH::V, BX = SH::BX;
    constexpr int ROWB = 16 * G * J;        // bytes per row: B float32 frames
    constexpr int U = DAS_PAIR_U;

    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint2 *lists = reinterpret_cast<uint2 *>(smem_raw);                     // [NP][LIST_STRIDE]
    float *dist_s = reinterpret_cast<float *>(lists + NP * LIST_STRIDE);    // [V][32]
    float2 *tx = reinterpret_cast<float2 *>(dist_s + V * MC);               // [V][Q]
    const int lane = threadIdx.x;

    const int bx = blockIdx.x % bricks_x;
    const int rb = blockIdx.x / bricks_x;
    const int by = rb % bricks_y;
    const int iz = g.nz - 1 - rb / bricks_y;
    const int KP = g.K + 3;
    auto voxel = [&](int v, int &n, float3 *pos) -> bool {
        if (g.vox) {
            n = blockIdx.x * V + v;
            if (n >= g.N) return false;
            if (pos) {
                const float4 p = __ldg(g.vox + n);
                *pos = make_float3(p.x, p.y, p.z);
            }
            n = voxel_index(g, n);
            return true;
        }
        const int ix = bx * BX + v % BX, iy = by * SH::BY + v / BX;
        if (ix >= g.nx || iy >= g.ny) return false;
        n = ix + g.nx * (iy + g.ny * iz);
        if (pos) *pos = voxel_position(g, ix, iy, iz);
        return true;
    };

    for (int e = lane; e < V * g.Q; e += 32) {
        const int v = e / g.Q, q = e % g.Q;
        float2 val = make_float2(0.f, 0.f);
        int n;
        if (voxel(v, n, nullptr)) {
            val.x = fmaf(__ldg(tau + (long long)q * g.N + n), g.fs, -g.t0fs);
            val.y = __ldg(wtx + (long long)q * g.N + n);
        }
        tx[e] = val;
    }
    // a non-finite sample anywhere in the record: single-voxel entries only
    const bool exact = nonfinite != nullptr && *(volatile const unsigned *)nonfinite != 0u;
    __syncwarp();

    const int grp = lane / G;               // this group's pair: voxels 2 grp, 2 grp + 1
    const int t = lane % G;                 // bytes [16 J t, 16 J (t + 1)) of every row
    const char *permB = reinterpret_cast<const char *>(perm) + t * 16 * J;
    const unsigned below = (1u << lane) - 1u;
    const float kmax = (float)(g.K - 1);
    const uint2 *ev = lists + grp * LIST_STRIDE;

    float2 accA[J][2], accB[J][2];
#pragma unroll
    for (int c = 0; c < J; ++c)
        accA[c][0] = accA[c][1] = accB[c][0] = accB[c][1] = make_float2(0.f, 0.f);
    // the third row of a window is loaded only when an offset needs it; its
    // registers keep earlier (finite) samples otherwise, times zero weights
    PTrip<U, J> ta, tb;
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
        for (int c = 0; c < J; ++c) ta.s[u][2][c] = tb.s[u][2][c] = make_uint4(0u, 0u, 0u, 0u);

    for (int m0 = 0; m0 < g.M; m0 += MC) {
        // ---- phase A: distances of the warp's voxels to receiver m0 + lane
        const int m = m0 + lane;
        const RxPos r = m < g.M ? __ldg(rx + m) : make_float4(0.f, 0.f, 0.f, 0.f);
        bool any = false;
#pragma unroll 4
        for (int i = 0; i < V; ++i) {
            float d = FAR;
            int n;
            float3 pos;
            if (m < g.M && voxel(i, n, &pos)) {
                float dd;
                if (receive_geometry(g, pos, r, dd)) {
                    d = dd;
                    any = true;
                }
            }
            dist_s[i * MC + lane] = d;
        }
        if (__ballot_sync(0xffffffffu, any) == 0u) continue;

        for (int q = q_begin; q < q_end; ++q) {
            const int base_row = (q * g.M + m0) * KP;
            // ---- phase B: the pairs' entry lists (the previous transmit's
            // phase C has finished reading them: __syncwarp below)
            int n_mine = 0;
#pragma unroll 2
            for (int p = 0; p < NP; ++p) {
                const float fA = tx[(2 * p) * g.Q + q].x + dist_s[(2 * p) * MC + lane];
                const float fB = tx[(2 * p + 1) * g.Q + q].x + dist_s[(2 * p + 1) * MC + lane];
                const float flA = floorf(fA), flB = floorf(fB);
                const bool okA = flA >= -1.f && flA <= kmax;    // false for NaN / inf / FAR
                const bool okB = flB >= -1.f && flB <= kmax;
                const bool both = okA && okB && !exact && fabsf(flA - flB) <= 1.f;
                const int cnt = both ? 1 : (int)okA + (int)okB;
                const unsigned b1 = __ballot_sync(0xffffffffu, cnt >= 1);
                const unsigned b2 = __ballot_sync(0xffffffffu, cnt >= 2);
                if (cnt >= 1) {
                    uint2 *L = lists + p * LIST_STRIDE + __popc(b1 & below) + __popc(b2 & below);
                    if (both) {
                        const float k = fminf(flA, flB);
                        L[0] = make_entry(lane * KP + (int)k + 1, fA - k, fB - k, 12u);
                    } else if (okA) {
                        L[0] = make_entry(lane * KP + (int)flA + 1, fA - flA, 0.f, 8u);
                        if (okB) L[1] = make_entry(lane * KP + (int)flB + 1, 0.f, fB - flB, 4u);
                    } else {
                        L[0] = make_entry(lane * KP + (int)flB + 1, 0.f, fB - flB, 4u);
                    }
                }
                if (p == grp) n_mine = __popc(b1) + __popc(b2);
            }
            __syncwarp();

            // ---- phase C
            const float wqA = tx[(2 * grp) * g.Q + q].y;
            const float wqB = tx[(2 * grp + 1) * g.Q + q].y;
            auto row_ptr = [&](unsigned x) {
                return permB + (long long)(base_row + (int)(x >> 4)) * ROWB;
            };
            if (!exact) {
                // entries i .. i + U - 1; those at or past the list's end are
                // neither read as rows nor used (their slots hold stale words)
                auto load_trip = [&](PTrip<U, J> &tr, int i) {
#pragma unroll
                    for (int u = 0; u < U; u += 2) {
                        if (u + 1 < U) {
                            const uint4 two = *reinterpret_cast<const uint4 *>(ev + i + u);
                            tr.e[u] = make_uint2(two.x, two.y);
                            tr.e[u + 1] = make_uint2(two.z, two.w);
                        } else {
                            tr.e[u] = ev[i + u];
                        }
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        if (i + u >= n_mine) {
                            tr.e[u] = make_uint2(0u, 0x80008000u);
                            continue;
                        }
                        const char *p0 = row_ptr(tr.e[u].x);
                        load_chunks<J>(p0, tr.s[u][0]);
                        load_chunks<J>(p0 + ROWB, tr.s[u][1]);
                        if (tr.e[u].x & 3u) load_chunks<J>(p0 + 2 * ROWB, tr.s[u][2]);
                    }
                };
                auto use_trip = [&](const PTrip<U, J> &tr, int nu) {
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        if (u >= nu) break;
                        const unsigned x = tr.e[u].x;
                        const float2 a = fractions(tr.e[u].y);
                        const float wA = (x & 8u) ? wqA : 0.f, wB = (x & 4u) ? wqB : 0.f;
                        const float uA = wA * a.x, vA = wA - uA;
                        const float uB = wB * a.y, vB = wB - uB;
                        const bool dA = x & 2u, dB = x & 1u;
                        const float cA0 = dA ? 0.f : vA, cA1 = dA ? vA : uA, cA2 = dA ? uA : 0.f;
                        const float cB0 = dB ? 0.f : vB, cB1 = dB ? vB : uB, cB2 = dB ? uB : 0.f;
#pragma unroll
                        for (int c = 0; c < J; ++c) {
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const float2 s0 = reinterpret_cast<const float2 *>(&tr.s[u][0][c])[h];
                                const float2 s1 = reinterpret_cast<const float2 *>(&tr.s[u][1][c])[h];
                                const float2 s2 = reinterpret_cast<const float2 *>(&tr.s[u][2][c])[h];
                                accA[c][h] = __ffma2_rn(make_float2(cA0, cA0), s0, accA[c][h]);
                                accA[c][h] = __ffma2_rn(make_float2(cA1, cA1), s1, accA[c][h]);
                                accA[c][h] = __ffma2_rn(make_float2(cA2, cA2), s2, accA[c][h]);
                                accB[c][h] = __ffma2_rn(make_float2(cB0, cB0), s0, accB[c][h]);
                                accB[c][h] = __ffma2_rn(make_float2(cB1, cB1), s1, accB[c][h]);
                                accB[c][h] = __ffma2_rn(make_float2(cB2, cB2), s2, accB[c][h]);
                            }
                        }
                    }
                };
                int i = 0;
                if (n_mine > 0) {
                    load_trip(ta, 0);
                    i = U;
                    for (;;) {
                        if (i >= n_mine) { use_trip(ta, n_mine - (i - U)); break; }
                        load_trip(tb, i);
                        i += U;
                        use_trip(ta, U);
                        if (i >= n_mine) { use_trip(tb, n_mine - (i - U)); break; }
                        load_trip(ta, i);
                        i += U;
                        use_trip(tb, U);
                    }
                }
            } else {
                // single-voxel entries, each added to its own voxel only
                for (int i = 0; i < n_mine; ++i) {
                    const uint2 e = ev[i];
                    const char *p0 = row_ptr(e.x);
                    const float2 a = fractions(e.y);
                    const bool isA = e.x & 8u;
                    const float w = isA ? wqA : wqB;
                    const float u1 = w * (isA ? a.x : a.y);
                    const float2 W0 = make_float2(w - u1, w - u1), W1 = make_float2(u1, u1);
                    uint4 r0[J], r1[J];
                    load_chunks<J>(p0, r0);
                    load_chunks<J>(p0 + ROWB, r1);
#pragma unroll
                    for (int c = 0; c < J; ++c) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const float2 s0 = reinterpret_cast<const float2 *>(&r0[c])[h];
                            const float2 s1 = reinterpret_cast<const float2 *>(&r1[c])[h];
                            float2 &acc = isA ? accA[c][h] : accB[c][h];
                            acc = __ffma2_rn(W1, s1, acc);
                            acc = __ffma2_rn(W0, s0, acc);
                        }
                    }
                }
            }
            // the next transmit rewrites the lists
            __syncwarp();
        }
    }

    // ---- write-out: lane t holds frames 4 (J t + c) .. + 3 of both voxels
#pragma unroll
    for (int vv = 0; vv < 2; ++vv) {
        int n;
        if (!voxel(2 * grp + vv, n, nullptr)) continue;
#pragma unroll
        for (int c = 0; c < J; ++c)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 a2 = vv ? accB[c][e >> 1] : accA[c][e >> 1];
                const float v = (e & 1) ? a2.y : a2.x;
                float *o = out + (long long)((J * t + c) * 4 + e) * g.N + n;
                *o = add_to_out ? *o + v : v;
            }
    }
}

template <int G, int J>
cudaError_t launch_one(const DasGeom &g, const RxPos *rx, const void *perm, const float *tau,
                       const float *w, float *out, const unsigned *nonfinite, cudaStream_t stream,
                       int q0, int q1, bool acc)
{
    using SH = PairShape<G>;
    const int bricks_x = g.vox ? (g.N + SH::V - 1) / SH::V : (g.nx + SH::BX - 1) / SH::BX;
    const int bricks_y = g.vox ? 1 : (g.ny + SH::BY - 1) / SH::BY;
    const long long blocks = (long long)bricks_x * bricks_y * (g.vox ? 1 : g.nz);
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const size_t smem = smem_bytes<G>(g.Q);
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    auto kernel = das_pair_kernel<G, J>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    kernel<<<(int)blocks, 32, smem, stream>>>(g, rx, perm, tau, w, out, bricks_x, bricks_y, nonfinite,
                                              q0, q1, acc ? 1 : 0);
    return cudaGetLastError();
}

// lanes per pair G and 16-byte chunks per lane J for B float32 frames: a lane
// holds 8 frames (one 256-bit load per row) where that leaves at least two
// lanes per pair, else 4
bool choose(int B, int &G, int &J)
{
    if ((B * 4) % 16 != 0) return false;
    const int cpr = B * 4 / 16;
#ifdef DAS_PAIR_FORCE_J1
    J = 1;
#else
    J = cpr >= 8 ? 2 : 1;
#endif
    G = cpr / J;
    return (G == 4 || G == 8) && G * J == cpr;
}

}  // namespace

bool pair_supported(int B, bool cplx, int K, bool half)
{
    int G, J;
    return !cplx && !half && K >= 2 && choose(B, G, J);
}

size_t pair_smem_bytes(int B, int Q)
{
    int G, J;
    if (!choose(B, G, J)) return 0;
    switch (G) {
    case 4: return smem_bytes<4>(Q);
    case 8: return smem_bytes<8>(Q);
    default: return smem_bytes<16>(Q);
    }
}

cudaError_t launch_pair(const DasGeom &g, const RxPos *rx, const void *perm, const float *tau,
                        const float *w, void *out, const unsigned *nonfinite, cudaStream_t stream,
                        int q0, int q1, bool accumulate)
{
    int G, J;
    if (q1 < 0) q1 = g.Q;
    if (q0 < 0 || q0 > q1 || q1 > g.Q) return cudaErrorInvalidValue;
    if (g.K < 2 || !choose(g.B, G, J)) return cudaErrorInvalidValue;
    float *o = static_cast<float *>(out);
#define DAS_PAIR_CASE(GG, JJ)                                                                   \
    if (G == GG && J == JJ)                                                                     \
        return launch_one<GG, JJ>(g, rx, perm, tau, w, o, nonfinite, stream, q0, q1, accumulate);
    DAS_PAIR_CASE(4, 1) DAS_PAIR_CASE(8, 1)
    DAS_PAIR_CASE(4, 2) DAS_PAIR_CASE(8, 2)
#undef DAS_PAIR_CASE
    return cudaErrorInvalidValue;
}

}  // namespace das
