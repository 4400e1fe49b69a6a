// WINDOW: this library's second sm_103a DAS kernel (not a design from the pages).
//
// What limits the brick kernel is the L1 data pipe: every 16-byte-per-lane
// load returns 512 bytes to registers in four wavefronts, and the four voxels
// of a warp mostly read the same or neighbouring sample rows, so about half of
// those bytes are duplicates.  This kernel makes one register load of a row
// serve several voxels:
//
//   * a group of G lanes (G * 16 bytes = one row of B float32 frames) owns a
//     quad of 2 x 2 neighbouring voxels (x, y) instead of one voxel;
//   * for one (transmit q, receiver m) the quad needs the rows k_j, k_j + 1 of
//     its four voxels j.  Neighbouring voxels lie within a few samples of each
//     other, so the union is a short window of rows lo .. hi + 1 (3.6 rows on
//     average for the 32 x 32-array volume instead of 8);
//   * each row of the window becomes one list entry: the row and four
//     coefficients, c_j = w(1 - a_j) on row k_j, w a_j on row k_j + 1, zero
//     elsewhere.  The group loads every row once and does y_j += c_j * s for
//     its four voxels (packed FP32 FMAs, two frames per instruction).
//
// Per warp: NQ = 32 / G quads.  Per pass of G receivers:
//   phase A (lane = (quad, receiver)): distance |x_j - r_m| in samples and the
//            F-number test for the quad's four voxels, in registers;
//   phase B (per transmit, same lanes): the window, its entries, and their
//            offsets in the quad's list by a prefix sum over the quad's lanes;
//            lists are padded to whole trips with zero entries on a zero row;
//   phase C: each group walks its quad's list, U entries per trip, the loads of
//            the next trip issued before the FMAs of the current one.
// A quad whose voxels are far apart in delay (a window of more than MAXE rows:
// arbitrary voxel lists) falls back to two entries per voxel.
//
// The record is the zero-padded layout Q x M x (K+3) x B of the brick kernel
// (sample k of slab (q, m) at row k + 1; rows 0, K+1, K+2 zero), so the window
// of a pair hanging over either end of the record reads zero rows.
#include "das_device.cuh"

#include <climits>

// tuning: warps per CTA, entries per phase-C trip, CTAs per SM the register
// allocation must allow (7: 72 registers, 28 warps; 32 x 32-array volume
// 14.9 ms, against 15.4 ms with 6 CTAs at 80 registers and 15.1 ms with 8 at 64)
#ifndef DAS_WINDOW_WARPS
#define DAS_WINDOW_WARPS 4
#endif
#ifndef DAS_WINDOW_U
#define DAS_WINDOW_U 4
#endif
#ifndef DAS_WINDOW_MIN_BLOCKS
#define DAS_WINDOW_MIN_BLOCKS 7
#endif

namespace das {
namespace {

constexpr int WARPS = DAS_WINDOW_WARPS;
constexpr int THREADS = 32 * WARPS;
constexpr int P = 4;                    // voxels per quad
constexpr int MAXE = 8;                 // list entries per (quad, receiver, transmit) at most
constexpr int U = DAS_WINDOW_U;         // entries per phase-C trip
constexpr float FAR = 1.0e30f;          // distance marking "outside the aperture"
constexpr int NOROW = -(1 << 28);       // row index of a voxel that takes no part

static_assert(U == 1 || U == 2 || U == 4, "trip size");

// Smallest n >= lo with n = r (mod m).
constexpr int round_up_mod(int lo, int m, int r) { return lo + ((r - lo % m) % m + m) % m; }

// Shapes for G lanes per quad: NQ quads per warp arranged QX x QY (each 2 x 2
// voxels), warps of a CTA arranged WGX x WGY, so a CTA covers BX x BY voxels
// of one x-y slice.  A quad list holds one pass (at most MAXE * G entries plus
// the padding to whole trips); its coefficient stride CAP and row stride CAPR
// put the lists of a warp's quads in different shared-memory banks.
template <int G>
struct Shape {
    static constexpr int NQ = 32 / G;
    static constexpr int QX = NQ >= 8 ? 4 : 2;
    static constexpr int QY = NQ / QX;
    static constexpr int WBX = 2 * QX, WBY = 2 * QY;
    static constexpr int WGX = WARPS >= 8 ? 4 : (WARPS >= 2 ? 2 : 1);   // warps of a CTA in x
    static constexpr int WGY = WARPS / WGX;
    static constexpr int BX = WBX * WGX, BY = WBY * WGY;
    static constexpr int V = NQ * P * WARPS;
    static constexpr int NEED = MAXE * G + U - 1;
    static constexpr int CAP = round_up_mod(NEED, 8, NQ == 4 ? 2 : 1);      // float4 entries
    static constexpr int CAPR = round_up_mod(NEED, 32, 4);                  // int entries
    static constexpr int ROWB = 16 * G;          // bytes per row: B = 4 G float32 frames
};

template <int G>
size_t smem_bytes(int Q)
{
    using S = Shape<G>;
    return (sizeof(float4) * S::CAP + sizeof(int) * S::CAPR) * (size_t)WARPS * S::NQ +
           sizeof(int) * 32 * WARPS + sizeof(float2) * (size_t)S::V * Q;
}

struct Trip {
    float4 c[U];
    uint4 s[U];
};

template <int G>
__global__ void __launch_bounds__(THREADS, DAS_WINDOW_MIN_BLOCKS)
das_window_kernel(DasGeom g, const RxPos *__restrict__ rx, const float *__restrict__ perm,
                  const float *__restrict__ tau, const float *__restrict__ wtx,
                  float *__restrict__ out, int bricks_x, int bricks_y, int q_begin, int q_end,
                  int add_to_out)
{
    using S = Shape<G>;
    constexpr int NQ = S::NQ;
    constexpr int CAP = S::CAP;
    constexpr int V = S::V;

    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int CAPR = S::CAPR;
    float4 *coef = reinterpret_cast<float4 *>(smem_raw);                  // [WARPS * NQ][CAP]
    int *rows = reinterpret_cast<int *>(coef + WARPS * NQ * CAP);         // [WARPS * NQ][CAPR]
    int *active = rows + WARPS * NQ * CAPR;                               // [WARPS][32]
    float2 *tx = reinterpret_cast<float2 *>(active + WARPS * 32);         // [V][Q]

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int quad = lane / G;
    const int t = lane % G;

    // brick (bx, by, iz), deepest slice first (deep voxels have the widest
    // apertures and the most work)
    const int bx = blockIdx.x % bricks_x;
    const int rb = blockIdx.x / bricks_x;
    const int by = rb % bricks_y;
    const int iz = g.nz - 1 - rb / bricks_y;
    const int KP = g.K + 3;

    // voxel v of this CTA, v = 4 (warp NQ + quad) + j: its index n (false if
    // the brick hangs over the grid or the list) and, on request, its position
    auto voxel = [&](int v, int &n, float3 *pos) -> bool {
        if (g.vox) {
            n = blockIdx.x * V + v;
            if (n >= g.N) return false;
            if (pos) {
                const float4 p = __ldg(g.vox + n);
                *pos = make_float3(p.x, p.y, p.z);
            }
            n = voxel_index(g, n);     // slot -> the caller's index
            return true;
        }
        const int j = v & 3, qd = (v >> 2) % NQ, w = (v >> 2) / NQ;
        const int ix = bx * S::BX + (w % S::WGX) * S::WBX + (qd % S::QX) * 2 + (j & 1);
        const int iy = by * S::BY + (w / S::WGX) * S::WBY + (qd / S::QX) * 2 + (j >> 1);
        if (ix >= g.nx || iy >= g.ny) return false;
        n = ix + g.nx * (iy + g.ny * iz);
        if (pos) *pos = voxel_position(g, ix, iy, iz);
        return true;
    };

    // ---- per-voxel transmit delay (samples) and weight, once per CTA
    for (int e = tid; e < V * g.Q; e += THREADS) {
        const int v = e / g.Q, q = e % g.Q;
        float2 val = make_float2(0.f, 0.f);
        int n;
        if (voxel(v, n, nullptr)) {
            val.x = fmaf(__ldg(tau + (long long)q * g.N + n), g.fs, -g.t0fs);
            val.y = __ldg(wtx + (long long)q * g.N + n);
        }
        tx[e] = val;
    }
    __syncthreads();

    const int vq = 4 * (warp * NQ + quad);            // first voxel of this lane's quad
    float4 *cq = coef + (warp * NQ + quad) * CAP;     // this quad's list
    int *rq = rows + (warp * NQ + quad) * CAPR;
    int *act = active + warp * 32;                    // this warp's active receivers
    const char *permB = reinterpret_cast<const char *>(perm) + t * 16;

    float2 acc[P][2];
#pragma unroll
    for (int j = 0; j < P; ++j) acc[j][0] = acc[j][1] = make_float2(0.f, 0.f);

    // lateral extent of this warp's voxel block (regular grid)
    const int ix0 = bx * S::BX + (warp % S::WGX) * S::WBX;
    const int iy0 = by * S::BY + (warp / S::WGX) * S::WBY;
    const float3 c0 = voxel_position(g, ix0, iy0, iz);
    const float3 c1 = voxel_position(g, ix0 + S::WBX - 1, iy0 + S::WBY - 1, iz);
    const float xlo = fminf(c0.x, c1.x), xhi = fmaxf(c0.x, c1.x);
    const float ylo = fminf(c0.y, c1.y), yhi = fmaxf(c0.y, c1.y);
    const unsigned below = (1u << lane) - 1u;

    for (int mb = 0; mb < g.M; mb += 32) {
        // ---- receivers mb + lane inside the aperture of some voxel of the
        // warp: the closest point of the block's lateral extent (grid; this
        // test passes whenever some voxel's exact test does), or each voxel
        // (list); compacted into act[0 .. nact)
        const int ml = mb + lane;
        bool in = false;
        if (ml < g.M) {
            const RxPos r = __ldg(rx + ml);
            if (!g.aperture) {
                in = true;
            } else if (g.vox) {
                for (int v = 4 * warp * NQ; v < 4 * (warp + 1) * NQ && !in; ++v) {
                    int n;
                    float3 pos;
                    if (voxel(v, n, &pos)) {
                        const float ex = pos.x - r.x, ey = pos.y - r.y, ez = pos.z - r.z;
                        in = ez > 0.f && g.ap2 * fmaf(ex, ex, ey * ey) <= ez * ez;
                    }
                }
            } else {
                const float ex = fmaxf(0.f, fmaxf(xlo - r.x, r.x - xhi));
                const float ey = fmaxf(0.f, fmaxf(ylo - r.y, r.y - yhi));
                const float ez = c0.z - r.z;
                in = ez > 0.f && g.ap2 * fmaf(ex, ex, ey * ey) <= ez * ez;
            }
        }
        const unsigned amask = __ballot_sync(0xffffffffu, in);
        if (amask == 0u) continue;
        if (in) act[__popc(amask & below)] = ml;
        __syncwarp();
        const int nact = __popc(amask);

        for (int p0 = 0; p0 < nact; p0 += G) {
            // ---- phase A: distances of the quad's voxels to active receiver p0 + t
            const int m = p0 + t < nact ? act[p0 + t] : -1;
            const RxPos r = m >= 0 ? __ldg(rx + m) : make_float4(0.f, 0.f, 0.f, 0.f);
            float dist[P];
            bool any = false;
#pragma unroll
            for (int j = 0; j < P; ++j) {
                dist[j] = FAR;
                int n;
                float3 pos;
                if (m >= 0 && voxel(vq + j, n, &pos)) {
                    float d;
                    if (receive_geometry(g, pos, r, d)) {
                        dist[j] = d;
                        any = true;
                    }
                }
            }
            if (__ballot_sync(0xffffffffu, any) == 0u) continue;

            for (int q = q_begin; q < q_end; ++q) {
                // ---- phase B: the window of rows of (q, m) for the quad
                const int slab = (q * g.M + m) * KP + 1;   // padded row of sample 0 (unused if m < 0)
                int k[P];
                float w0[P], w1[P];
                int lo = INT_MAX, hi = INT_MIN, nok = 0;
#pragma unroll
                for (int j = 0; j < P; ++j) {
                    const float2 tj = tx[(vq + j) * g.Q + q];
                    const float f = tj.x + dist[j];
                    const float fl = floorf(f);
                    // inside the aperture (dist < FAR) and a sample inside the
                    // record; false for NaN / inf
                    const bool ok = (fl >= -1.f) && (fl <= (float)(g.K - 1));
                    const float a = f - fl;
                    w1[j] = tj.y * a;
                    w0[j] = tj.y - w1[j];
                    k[j] = ok ? (int)fl : NOROW;
                    if (ok) {
                        lo = min(lo, k[j]);
                        hi = max(hi, k[j]);
                        ++nok;
                    }
                }
                const bool win = nok > 0 && hi - lo <= MAXE - 2;
                const int nent = nok == 0 ? 0 : (win ? hi - lo + 2 : 2 * nok);
                // offsets in the quad's list: prefix sum over the quad's G lanes
                int incl = nent;
#pragma unroll
                for (int s = 1; s < G; s <<= 1) {
                    const int o = __shfl_up_sync(0xffffffffu, incl, s, G);
                    if (t >= s) incl += o;
                }
                const int total = __shfl_sync(0xffffffffu, incl, G - 1, G);
                int pos = incl - nent;
                if (win) {
                    for (int e = 0; e < nent; ++e) {
                        const int R = lo + e;
                        float c[P];
#pragma unroll
                        for (int j = 0; j < P; ++j)
                            c[j] = k[j] == R ? w0[j] : (k[j] + 1 == R ? w1[j] : 0.f);
                        cq[pos + e] = make_float4(c[0], c[1], c[2], c[3]);
                        rq[pos + e] = slab + R;
                    }
                } else if (nok > 0) {
                    // voxels far apart in delay: rows k_j, k_j + 1 of each voxel
#pragma unroll
                    for (int j = 0; j < P; ++j) {
                        if (k[j] == NOROW) continue;
                        float c0[P], c1[P];
#pragma unroll
                        for (int i = 0; i < P; ++i) {
                            c0[i] = i == j ? w0[j] : 0.f;
                            c1[i] = i == j ? w1[j] : 0.f;
                        }
                        cq[pos] = make_float4(c0[0], c0[1], c0[2], c0[3]);
                        rq[pos] = slab + k[j];
                        cq[pos + 1] = make_float4(c1[0], c1[1], c1[2], c1[3]);
                        rq[pos + 1] = slab + k[j] + 1;
                        pos += 2;
                    }
                }
                // pad to whole trips: zero coefficients on row 0, a zero row
                const int padded = (total + U - 1) / U * U;
                if (t == G - 1)
                    for (int e = total; e < padded; ++e) {
                        cq[e] = make_float4(0.f, 0.f, 0.f, 0.f);
                        rq[e] = 0;
                    }
                __syncwarp();

                // ---- phase C: this group's list, U entries per trip, pipelined
                const int ntrips = padded / U;
                auto load_trip = [&](Trip &tr, int i) {
                    int rr[U];
                    if constexpr (U == 4) {
                        const int4 v4 = *reinterpret_cast<const int4 *>(rq + i);
                        rr[0] = v4.x; rr[1] = v4.y; rr[2] = v4.z; rr[3] = v4.w;
                    } else if constexpr (U == 2) {
                        const int2 v2 = *reinterpret_cast<const int2 *>(rq + i);
                        rr[0] = v2.x; rr[1] = v2.y;
                    } else {
                        rr[0] = rq[i];
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        tr.c[u] = cq[i + u];
                        tr.s[u] = __ldg(reinterpret_cast<const uint4 *>(permB + (long long)rr[u] * S::ROWB));
                    }
                };
                auto use_trip = [&](const Trip &tr) {
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const float2 s01 = make_float2(__uint_as_float(tr.s[u].x), __uint_as_float(tr.s[u].y));
                        const float2 s23 = make_float2(__uint_as_float(tr.s[u].z), __uint_as_float(tr.s[u].w));
                        const float c[P] = {tr.c[u].x, tr.c[u].y, tr.c[u].z, tr.c[u].w};
#pragma unroll
                        for (int j = 0; j < P; ++j) {
                            const float2 cc = make_float2(c[j], c[j]);
                            acc[j][0] = __ffma2_rn(cc, s01, acc[j][0]);
                            acc[j][1] = __ffma2_rn(cc, s23, acc[j][1]);
                        }
                    }
                };
                if (ntrips > 0) {
                    Trip ta, tb;
                    load_trip(ta, 0);
                    int i = 1;
                    for (;;) {
                        if (i >= ntrips) { use_trip(ta); break; }
                        load_trip(tb, i * U);
                        ++i;
                        use_trip(ta);
                        if (i >= ntrips) { use_trip(tb); break; }
                        load_trip(ta, i * U);
                        ++i;
                        use_trip(tb);
                    }
                }
                __syncwarp();   // the list is rewritten for the next transmit
            }
        }
        __syncwarp();       // act is rewritten for the next block
    }

    // ---- y[b, n] for the quad's voxels, frames b = 4 t .. 4 t + 3
#pragma unroll
    for (int j = 0; j < P; ++j) {
        int n;
        if (!voxel(vq + j, n, nullptr)) continue;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const long long idx = (long long)(4 * t + e) * g.N + n;
            const float v = (e & 1) ? acc[j][e >> 1].y : acc[j][e >> 1].x;
            out[idx] = add_to_out ? out[idx] + v : v;
        }
    }
}

template <int G>
cudaError_t launch_g(const DasGeom &g, const RxPos *rx, const void *perm, const float *tau,
                     const float *w, float *out, cudaStream_t stream, int q0, int q1, bool acc)
{
    using S = Shape<G>;
    const int bricks_x = g.vox ? (g.N + S::V - 1) / S::V : (g.nx + S::BX - 1) / S::BX;
    const int bricks_y = g.vox ? 1 : (g.ny + S::BY - 1) / S::BY;
    const long long blocks = (long long)bricks_x * bricks_y * (g.vox ? 1 : g.nz);
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const size_t smem = smem_bytes<G>(g.Q);
    auto kernel = das_window_kernel<G>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    kernel<<<(int)blocks, THREADS, smem, stream>>>(g, rx, static_cast<const float *>(perm), tau, w, out,
                                                   bricks_x, bricks_y, q0, q1, acc ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace

bool window_supported(int B, bool cplx, int K, int Q, int M, bool half)
{
    if (cplx || half || K < 2 || Q < 0) return false;
    size_t smem;
    switch (B) {
    case 32: smem = smem_bytes<8>(Q); break;
    case 16: smem = smem_bytes<4>(Q); break;
    case 8: smem = smem_bytes<2>(Q); break;
    default: return false;
    }
    // the lists and transmit table fit one CTA's shared memory, and absolute
    // padded row indices fit 32 bits
    return smem <= 227u * 1024u && (long long)Q * M * (K + 3) < 0x7fffffffLL;
}

cudaError_t launch_window(const DasGeom &g, const RxPos *rx, const void *perm, const float *tau,
                          const float *w, void *out, cudaStream_t stream, int q0, int q1,
                          bool accumulate)
{
    if (q1 < 0) q1 = g.Q;
    if (q0 < 0 || q0 > q1 || q1 > g.Q) return cudaErrorInvalidValue;
    if (!window_supported(g.B, false, g.K, g.Q, g.M, false)) return cudaErrorInvalidValue;
    float *o = static_cast<float *>(out);
    switch (g.B) {
    case 32: return launch_g<8>(g, rx, perm, tau, w, o, stream, q0, q1, accumulate);
    case 16: return launch_g<4>(g, rx, perm, tau, w, o, stream, q0, q1, accumulate);
    case 8: return launch_g<2>(g, rx, perm, tau, w, o, stream, q0, q1, accumulate);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace das
