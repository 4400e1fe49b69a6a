// BRICK: this library's DAS kernel for sm_103a (not a design from the pages).
//
// Each CTA (WARPS warps, one by default) owns a brick of V voxels in one x-y
// slice (4 x 1 for 32 frames of float32 with one warp) and all B frames of
// them.  Neighbouring voxels of a slice need nearly the same sample rows of
// every receiver, so the groups of a warp walking the same receivers at the
// same time hit the same L1 lines; bricks are flat in z because one voxel step
// in depth moves the delay by many samples.  One-warp CTAs measured fastest
// (32-frame float32 volume: 8 warps 13.8 ms, 4 13.2, 2 13.0, 1 12.5): the
// transmit-delay preload needs no CTA-wide barrier wait, and the scheduler
// balances finer pieces of work.
//
// The record is permuted to the zero-padded layout Q x M x (K+3) x B (sample k
// of slab (q, m) at row k + 1, rows 0, K+1, K+2 zero), so the two rows a voxel
// reads for a (q, m) are adjacent and a pair that hangs over either end of the
// record reads a zero row instead of needing special weights.  A group of G
// lanes owns one voxel and reads the voxel's two rows in 16-byte chunks:
//   pair mode  : lane t loads chunks t, t + G, ... of both rows (float32 data,
//                and half-precision rows of more than 64 bytes); G = 8 lanes
//                cover one 128-byte line per row (16 lanes two lines);
//   split mode : half-precision rows of at most 64 bytes: the 2 * CPR chunks of
//                the two adjacent rows go one per lane (G = 2 * CPR), so a group
//                reads one contiguous run; the partial sums of the two rows are
//                added by one shuffle at the end.
// Half-precision samples are converted to float32 before the interpolation
// and the accumulation (ffdas paper, Methods, FP16 paragraphs).
//
// A warp owns NW = 32 / G voxels and does all the work for them itself, so
// after the per-CTA preload of transmit delays no step needs a CTA barrier:
//   phase A (per block of 32 receivers, lane = receiver): distance |x_v - r_m|
//            in samples and the F-number test for the warp's NW voxels, kept in
//            registers; a block whose receivers lie outside every aperture of
//            the warp's voxels is skipped.  A brick starts its walk over the
//            blocks at the one its co-resident bricks have reached (its CTA
//            index over the CTAs resident at once), so that they spread over
//            the record's slabs;
//   phase B (per transmit, lane = receiver): an entry for every pair that
//            contributes (inside the voxel's aperture, a sample inside the
//            record), in aligned lists in the warp's own shared memory: a warp
//            ballot over "some voxel of the warp contributes" gives each such
//            receiver one slot in every voxel's list, so the groups read rows of
//            the same slab in each instruction and share L1 lines; a voxel
//            without a term for that receiver reads the slab's zero pad rows.
//            Lists are double-buffered by transmit parity (entry formats below);
//   phase C: each group walks its voxel's list U entries per trip, software
//            pipelined: the row loads of the next trip are issued before the
//            FMAs of the current one, so a warp keeps two trips of loads in
//            flight; with aligned lists the groups walk in step.  Real data are
//            accumulated two frames at a time with the packed FP32 FMA of
//            sm_100+ (__ffma2_rn), halving the FMA instructions; the two rows'
//            weights come from the entry with one FMA and one subtraction (the
//            fraction read in place as mantissa bits, the transmit weight scaled
//            to match), complex ones from the entry's weighted phase.
// The host side may split the transmits (and the receivers) over several
// launches that add to y, so that the record rows in use at one time fit L2.
#include <cuda_fp16.h>

#include <cmath>

#include "das_device.cuh"

// tuning (one chunk per lane, float32 or half storage): receivers per
// phase-C trip and the warps per SM the register allocation must allow; and
// the warps per CTA
#ifndef DAS_BRICK_U1
#define DAS_BRICK_U1 4
#endif
#ifndef DAS_BRICK_MIN_WARPS
#define DAS_BRICK_MIN_WARPS 32
#endif
#ifndef DAS_BRICK_WARPS
#define DAS_BRICK_WARPS 1
#endif
#ifndef DAS_BRICK_PACKED
#define DAS_BRICK_PACKED 1     // real entries packed into 32 bits (else {row, fraction} floats)
#endif
// 4 lanes x 8 frames per voxel (one 256-bit load per row and lane) for rows of
// 128 bytes, instead of 8 lanes x 4 frames; its warps per SM and trip size
#ifndef DAS_BRICK_CONTIG_B32
#define DAS_BRICK_CONTIG_B32 0
#endif
#ifndef DAS_BRICK_C_WARPS
#define DAS_BRICK_C_WARPS 24
#endif
#ifndef DAS_BRICK_C_U
#define DAS_BRICK_C_U 2
#endif
// aligned lists: slot s of every voxel's list belongs to the s-th receiver of
// the block that contributes to some voxel of the warp, so the groups load rows
// of one slab at the same time; where a voxel has no term for that receiver its
// entry reads the slab's two zero pad rows (K+1, K+2) and adds exactly zero
// (0: lists compacted per voxel, the form before)
#ifndef DAS_BRICK_ALIGNED
#define DAS_BRICK_ALIGNED 1
#endif
// rotated receiver loop: a brick starts its walk over the blocks of receivers
// at the block the bricks resident with it have reached (percent of one wave
// of resident CTAs per lap; 0: every brick starts at the first block)
#ifndef DAS_BRICK_ROT
#define DAS_BRICK_ROT 100
#endif
// complex64 rows of 64 frames (16 lanes x 2 chunks): two packed accumulators
// per sample, one for the real and one for the imaginary part of the weight
// (four packed FMAs per complex sample and entry instead of eight scalar ones;
// 24 warps per SM for the registers); 0: complex FMAs.  Half2 storage keeps the
// complex FMAs (fewer registers, more warps: faster there)
#ifndef DAS_BRICK_CSPLIT
#define DAS_BRICK_CSPLIT 1
#endif
// real float entries carry the weight w a of the second row instead of the
// fraction a (phase B multiplies once per voxel and receiver, not each lane)
#ifndef DAS_BRICK_WENTRY
#define DAS_BRICK_WENTRY 1
#endif
// packed entries: the fraction decoded as 1 + a (a float in [1, 2)) and the
// weight of the second row taken as wq (1 + a) - wq in one FMA
#ifndef DAS_BRICK_FOLD
#define DAS_BRICK_FOLD 1
#endif
// packed entries: the fraction bits read in place as the low mantissa bits of
// a float in [1, 2) (one masked OR), the transmit weight scaled by 2^(23 - fb)
// complex entries carry the transmit weight times the demodulation phase, so
// phase C forms the two complex weights with 2 multiplies and 2 subtractions
#ifndef DAS_BRICK_IQPRE
#define DAS_BRICK_IQPRE 1
#endif
// preferred shared-memory carveout in percent of the SM's unified L1 / shared
// array (-1: the driver's choice), raised where the CTAs the launch bounds ask
// for need more.  Measured on the 32-frame float32 volume: 11.19 ms at 44 %
// (a 200.7 KB shared configuration, by the profiler) against 11.41 ms with the
// driver's choice (102.4 KB) and 12.56 ms at 58 % or more
#ifndef DAS_BRICK_CARVEOUT
#define DAS_BRICK_CARVEOUT 44
#endif
#ifndef DAS_BRICK_LOWFRAC
#define DAS_BRICK_LOWFRAC 1
#endif

namespace das {
namespace {

constexpr int WARPS = DAS_BRICK_WARPS;   // warps per CTA (= per brick)
constexpr int THREADS = 32 * WARPS;
constexpr int MC = 32;                 // receivers per block (one per lane in phases A and B)
constexpr float FAR = 1.0e30f;         // distance marking "outside the aperture"

// brick footprint in x (voxels), as square as powers of two allow; the
// footprint in y is V / BX (DAS_BRICK_BX: a fixed footprint in x where it
// divides V)
#ifndef DAS_BRICK_BX
#define DAS_BRICK_BX 0
#endif
template <int V>
struct BrickShape {
    static constexpr int BX = (DAS_BRICK_BX > 0 && V % (DAS_BRICK_BX > 0 ? DAS_BRICK_BX : 1) == 0)
                                  ? (DAS_BRICK_BX > V ? V : DAS_BRICK_BX)
                                  : (V >= 512 ? 32 : (V >= 128 ? 16 : (V >= 32 ? 8 : (V >= 4 ? 4 : V))));
    static_assert(V >= 1 && (V & (V - 1)) == 0 && V % BX == 0, "bricks tile V voxels");
};

// Real entry: one 32-bit word, the row relative to the first row of the block
// of receivers in the high bits and the interpolation fraction, rounded to
// nearest (at most 1 - 2^-FB), in the low FB bits (FB >= 10; for K = 2048, 15 bits, a step of 3e-5
// samples, 8x finer than float32 resolves f near K; for K = 65536, 10 bits, a
// step of 1e-3 samples, half the float32 resolution of f there) -- or {row,
// fraction} in float32 bits.
// IQ entry: {row, fraction, cos, sin} in float32 bits.  Real entries are
// packed for float32 storage, whose phase C is bound by shared-memory and L1
// traffic, while at least MIN_PACKED_BITS fraction bits remain (K <= 8189);
// longer records (WIDE) and half storage keep the undecoded floats.
constexpr int MIN_PACKED_BITS = 14;
template <bool CPLX, bool HALF, bool WIDE>
constexpr bool packed_entries() { return !CPLX && !HALF && !WIDE && DAS_BRICK_PACKED != 0; }
template <bool CPLX, bool HALF, bool WIDE>
using Entry = typename std::conditional<CPLX, float4,
                                        typename std::conditional<packed_entries<CPLX, HALF, WIDE>(),
                                                                  unsigned, float2>::type>::type;

// entries per voxel list: MC plus padding, so that a list starts on a 16-byte
// boundary and the lists of a warp's voxels start in different banks
template <bool CPLX>
constexpr int entry_stride() { return CPLX ? MC + 1 : MC + 2; }

// fraction bits of a packed entry for records of K samples: the relative row
// (< 32 (K + 3)) takes the high bits, the fraction the rest (at most 23)
inline int fraction_bits(int K)
{
    const long long span = 32LL * (K + 3);
    int rel_bits = 0;
    while ((1LL << rel_bits) < span) ++rel_bits;
    const int fb = 32 - rel_bits;
    return fb > 23 ? 23 : fb;
}

// Storage of the permuted record as seen by one lane of a group.
//   EPC  elements per 16-byte chunk (float32 4, complex64 2, half 8, half2 4)
//   ROWB bytes per row (B * element size)
//   L    16-byte loads per entry and lane
//   NA   accumulator chunks per lane
//   NP   float2 accumulators per chunk (real: frame pairs; IQ: one per frame)
template <int G, int J, bool CPLX, bool HALF, bool SPLIT>
struct Layout {
    static constexpr int ESZ = HALF ? (CPLX ? 4 : 2) : (CPLX ? 8 : 4);
    static constexpr int EPC = 16 / ESZ;
    static constexpr int ROWB = SPLIT ? 8 * G : 16 * G * J;
    static constexpr int L = SPLIT ? 1 : 2 * J;
    static constexpr int NA = SPLIT ? 1 : J;
    static constexpr int NP = CPLX ? EPC : EPC / 2;
};

template <int G, bool CPLX, bool HALF, bool WIDE>
size_t smem_bytes(int Q)
{
    constexpr int V = WARPS * (32 / G);
    return sizeof(Entry<CPLX, HALF, WIDE>) * 2 * V * entry_stride<CPLX>() + sizeof(float2) * (size_t)V * Q;
}

// One pipelined trip of phase C: U entries, their fractions (and phases) and
// the L chunks of each.
template <int U, int L>
struct Trip {
    float a[U];
    float2 ph[U];
    uint4 s[U][L];
};

// two adjacent 16-byte chunks in one 256-bit load
__device__ __forceinline__ void load256(const char *p, uint4 &a, uint4 &b)
{
    asm("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
        : "l"(p));
}

// 16 bytes of samples -> NP float2 values: pairs of consecutive frames (real)
// or one complex sample each (IQ), in float32
template <bool HALF, int NP>
__device__ __forceinline__ void unpack(uint4 u, float2 (&v)[NP])
{
    if constexpr (HALF) {
        const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
        for (int i = 0; i < NP; ++i) v[i] = __half22float2(h[i]);
    } else {
        const float2 *p = reinterpret_cast<const float2 *>(&u);
#pragma unroll
        for (int i = 0; i < NP; ++i) v[i] = p[i];
    }
}

// acc += w * s: real frame pairs with one packed FMA, complex with four FMAs
template <bool CPLX>
__device__ __forceinline__ void mac(float2 &acc, float2 w, float2 s)
{
    if constexpr (CPLX) cfma(acc, w, s);
    else acc = __ffma2_rn(w, s, acc);
}

// acc += w0 * (row-0 chunks) + w1 * (row-1 chunks), w1 = wq * fraction,
// w0 = wq - w1 (IQ: both weights rotated by the entry's phase; real: the
// weight broadcast to both frames of a pair).  In split mode the lane holds
// one chunk of row `split_row`.  With split complex accumulators, acc[c][e]
// collects w Re(ph) s and acc[c][NP + e] collects w Im(ph) s, each with
// packed FMAs on (Re s, Im s); the output is the first plus i times the second.
template <int G, int J, bool CPLX, bool HALF>
constexpr bool split_complex() { return CPLX && !HALF && G == 16 && J == 2 && DAS_BRICK_CSPLIT != 0; }

// Weight of the second row from an entry's number a: WM 0, a is the fraction
// (w1 = wq a); WM 1, a is w1 itself; WM 2, a is 1 + the fraction, so
// w1 = wq (1 + fraction) - wq in one FMA, the same rounding of the same exact
// product as wq * fraction; WM 3, a is 1 + the fraction's bits times 2^-23
// and wqs = wq 2^(23 - fb), so w1 = wqs a - wqs, again the same product.
template <bool CPLX, bool HALF, bool SPLIT, int WM, bool CS, int NA, int NPA, int L>
__device__ __forceinline__ void accumulate(float2 (&acc)[NA][NPA], float wq, float wqs, float a,
                                           float2 ph, const uint4 (&s)[L], int split_row)
{
    constexpr int NP = CS ? NPA / 2 : NPA;
    const float w1 = WM == 1 ? a : (WM == 2 ? fmaf(wq, a, -wq) : (WM == 3 ? fmaf(wqs, a, -wqs) : wq * a));
    const float w0 = wq - w1;
    // complex, WM 4: the entry's phase is already w exp(i phi), so the second
    // row's complex weight is a times it and the first row's the rest
    const float c1 = WM == 4 ? a * ph.x : w1 * ph.x, s1 = WM == 4 ? a * ph.y : w1 * ph.y;
    const float c0 = WM == 4 ? ph.x - c1 : w0 * ph.x, s0 = WM == 4 ? ph.y - s1 : w0 * ph.y;
    if constexpr (CS) {
        const float2 R0 = make_float2(c0, c0), I0 = make_float2(s0, s0);
        const float2 R1 = make_float2(c1, c1), I1 = make_float2(s1, s1);
        if constexpr (SPLIT) {
            const float2 R = split_row ? R1 : R0, I = split_row ? I1 : I0;
            float2 v[NP];
            unpack<HALF, NP>(s[0], v);
#pragma unroll
            for (int e = 0; e < NP; ++e) {
                acc[0][e] = __ffma2_rn(R, v[e], acc[0][e]);
                acc[0][NP + e] = __ffma2_rn(I, v[e], acc[0][NP + e]);
            }
        } else {
#pragma unroll
            for (int c = 0; c < NA; ++c) {
                float2 v0[NP], v1[NP];
                unpack<HALF, NP>(s[2 * c], v0);
                unpack<HALF, NP>(s[2 * c + 1], v1);
#pragma unroll
                for (int e = 0; e < NP; ++e) {
                    acc[c][e] = __ffma2_rn(R1, v1[e], acc[c][e]);
                    acc[c][e] = __ffma2_rn(R0, v0[e], acc[c][e]);
                    acc[c][NP + e] = __ffma2_rn(I1, v1[e], acc[c][NP + e]);
                    acc[c][NP + e] = __ffma2_rn(I0, v0[e], acc[c][NP + e]);
                }
            }
        }
        return;
    }
    const float2 W0 = CPLX ? make_float2(c0, s0) : make_float2(w0, w0);
    const float2 W1 = CPLX ? make_float2(c1, s1) : make_float2(w1, w1);
    if constexpr (SPLIT) {
        const float2 W = split_row ? W1 : W0;
        float2 v[NP];
        unpack<HALF, NP>(s[0], v);
#pragma unroll
        for (int e = 0; e < NP; ++e) mac<CPLX>(acc[0][e], W, v[e]);
    } else {
#pragma unroll
        for (int c = 0; c < NA; ++c) {
            float2 v0[NP], v1[NP];
            unpack<HALF, NP>(s[2 * c], v0);
            unpack<HALF, NP>(s[2 * c + 1], v1);
#pragma unroll
            for (int e = 0; e < NP; ++e) {
                mac<CPLX>(acc[c][e], W1, v1[e]);
                mac<CPLX>(acc[c][e], W0, v0[e]);
            }
        }
    }
}

// Warps per SM the register allocation must allow: lanes that hold more
// chunks (J) or complex samples keep more row data in flight per trip, so
// they get fewer warps (more registers each); 16-lane groups (at most two
// chunks a lane) fit 32 warps, 24 for complex with 4 entries per trip.  The
// CTA count per SM is that over the warps per CTA.
// A lane that holds its J chunks contiguously (4 lanes x 2 chunks: one 256-bit
// load per row, so a group still reads one full 128-byte line per row).
template <int G, int J, bool CPLX, bool HALF>
constexpr bool contiguous_chunks() { return G == 4 && J == 2 && !CPLX && !HALF; }

// (split complex accumulators on 16 lanes x 2 chunks: 24 warps, 80 registers)
// MWO > 0 overrides the count: the 4-lane float32 layout runs at 28 warps (72
// registers) when the record fits in L2 (16 frames, 5 x 256 slabs: 0.506 against
// 0.516 ms; on records that stream from DRAM 28 warps lose 4 %)
template <int G, int J, bool CPLX, bool HALF, int MWO = 0>
constexpr int min_warps()
{
    return MWO > 0 ? MWO
         : contiguous_chunks<G, J, CPLX, HALF>()
               ? DAS_BRICK_C_WARPS
               : G == 16 ? ((CPLX && J == 1) || split_complex<G, J, CPLX, HALF>() ? 24 : 32)
                         : (J >= 4 ? 16 : (J == 2 || CPLX ? 24 : DAS_BRICK_MIN_WARPS));
}
template <int G, int J, bool CPLX, bool HALF, int MWO = 0>
constexpr int min_blocks()
{
    // at least 1, at most the 32 resident CTAs an SM holds
    return min_warps<G, J, CPLX, HALF, MWO>() / WARPS < 1
               ? 1
               : (min_warps<G, J, CPLX, HALF, MWO>() / WARPS > 32 ? 32
                                                                  : min_warps<G, J, CPLX, HALF, MWO>() / WARPS);
}
#ifndef DAS_BRICK_L2_WARPS_G4
#define DAS_BRICK_L2_WARPS_G4 28
#endif

// receivers per phase-C trip
template <int G, int J, bool CPLX, bool HALF>
constexpr int trip_size()
{
    return contiguous_chunks<G, J, CPLX, HALF>() ? DAS_BRICK_C_U
                                                 : (J >= 4 ? 1 : (J == 2 ? 2 : DAS_BRICK_U1));
}

template <int G, int J, bool CPLX, bool HALF, bool SPLIT, bool WIDE, int MWO>
__global__ void __launch_bounds__(THREADS, min_blocks<G, J, CPLX, HALF, MWO>())
das_brick_kernel(DasGeom g, const RxPos *__restrict__ rx, const void *__restrict__ perm,
                 const float *__restrict__ tau, const float *__restrict__ wtx,
                 float *__restrict__ out, int bricks_x, int bricks_y, int fb, int q_begin,
                 int q_end, int m_begin, int m_end, int add_to_out, long long rot_wave)
{
    using LY = Layout<G, J, CPLX, HALF, SPLIT>;
    constexpr int NW = 32 / G;                     // voxels per warp
    constexpr int V = WARPS * NW;                  // voxels per CTA
    constexpr int BX = BrickShape<V>::BX;
    constexpr int EPC = LY::EPC;
    constexpr int NP = LY::NP;
    constexpr int L = LY::L;
    constexpr int NA = LY::NA;
    constexpr int ROWB = LY::ROWB;
    constexpr int CPR = ROWB / 16;                 // 16-byte chunks per row
    constexpr int U = trip_size<G, J, CPLX, HALF>();   // receivers per loop trip
    constexpr bool CONTIG = contiguous_chunks<G, J, CPLX, HALF>();
    constexpr int ES = entry_stride<CPLX>();
    using E = Entry<CPLX, HALF, WIDE>;
    constexpr bool PACKED = packed_entries<CPLX, HALF, WIDE>();
    constexpr bool PRE = !CPLX && !PACKED && DAS_BRICK_WENTRY != 0;   // entries hold w a
    constexpr bool FOLD = !CPLX && PACKED && DAS_BRICK_FOLD != 0;     // decode gives 1 + a
    constexpr bool LOWF = FOLD && DAS_BRICK_LOWFRAC != 0;            // fraction bits kept low
    constexpr bool CPRE = CPLX && DAS_BRICK_IQPRE != 0;               // IQ entries hold w exp(i phi)
    constexpr int WM = CPRE ? 4 : (PRE ? 1 : (LOWF ? 3 : (FOLD ? 2 : 0)));

    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    E *ent = reinterpret_cast<E *>(smem_raw) + warp * (2 * NW * ES);        // this warp's [2][NW][ES]
    float2 *tx = reinterpret_cast<float2 *>(reinterpret_cast<E *>(smem_raw) + 2 * V * ES);  // [V][Q]

    // Grid: brick (bx, by, iz), deepest slice first (deep voxels have the
    // widest apertures and the most work, so launching them first leaves the
    // light shallow bricks for the tail).  Voxel list: V consecutive entries.
    const int bx = blockIdx.x % bricks_x;
    const int rb = blockIdx.x / bricks_x;
    const int by = rb % bricks_y;
    const int iz = g.nz - 1 - rb / bricks_y;
    const int KP = g.K + 3;                        // rows per padded slab
    // voxel v of this CTA: its index n (false if the brick hangs over the grid
    // or the list) and, on request, its position in sample units
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
        const int ix = bx * BX + v % BX, iy = by * (V / BX) + v / BX;
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

    // ---- this warp's voxels v0 + i, i < NW; group grp consumes voxel v0 + grp
    const int v0 = warp * NW;
    const int grp = lane / G;
    const int t = lane % G;
    // pair mode: load 2c + r of a lane is chunk t + G c of row r; split mode: the
    // lane's one load is chunk t of the row pair (row t / CPR)
    const char *permB = reinterpret_cast<const char *>(perm) + t * 16 * (CONTIG ? J : 1);
    const int split_row = SPLIT ? t / CPR : 0;
    const unsigned below = (1u << lane) - 1u;
    const unsigned frac_mask = (1u << fb) - 1u;
    const float frac_scale = (float)(1u << fb);
    const unsigned frac_shift = 23u - (unsigned)fb;   // fraction bits -> top of a float mantissa
    const float frac_pow = (float)(1u << frac_shift);

    constexpr bool CS = split_complex<G, J, CPLX, HALF>();
    constexpr int NPA = CS ? 2 * NP : NP;   // accumulators per chunk
    float2 acc[NA][NPA];
#pragma unroll
    for (int c = 0; c < NA; ++c)
#pragma unroll
        for (int e = 0; e < NPA; ++e) acc[c][e] = make_float2(0.f, 0.f);

    const int n_blocks = (m_end - m_begin + MC - 1) / MC;
    const int b_first = rot_wave > 0 ? (int)(((long long)blockIdx.x * n_blocks / rot_wave) % n_blocks) : 0;
    for (int bi = 0; bi < n_blocks; ++bi) {
        int b = bi + b_first;
        if (b >= n_blocks) b -= n_blocks;
        const int m0 = m_begin + MC * b;
        // ---- phase A: distances of the warp's voxels to receiver m0 + lane
        const int m = m0 + lane;
        const RxPos r = m < g.M ? __ldg(rx + m) : make_float4(0.f, 0.f, 0.f, 0.f);
        float dist[NW];
        bool any = false;
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            dist[i] = FAR;
            int n;
            float3 pos;
            if (m < g.M && voxel(v0 + i, n, &pos)) {
                float d;
                if (receive_geometry(g, pos, r, d)) {
                    dist[i] = d;
                    any = true;
                }
            }
        }
        if (__ballot_sync(0xffffffffu, any) != 0u) {
            for (int q = q_begin; q < q_end; ++q) {
                E *eb = ent + (q & 1) * NW * ES;
                // ---- phase B: compacted entry lists of the warp's voxels
                int n_mine = 0;
                const int base_row = (q * g.M + m0) * KP;    // row 0 of this block's first slab
                // the entry of voxel i for this lane's receiver
                auto make = [&](float f, float fl, float wv) -> E {
                    const int rel = lane * KP + (int)fl + 1;  // row within this block
                    const float a = f - fl;                   // in [0, 1)
                    if constexpr (CPLX) {
                        const float2 ph = demod_phase(g, f);
                        return CPRE ? make_float4(__int_as_float(base_row + rel), a, wv * ph.x, wv * ph.y)
                                    : make_float4(__int_as_float(base_row + rel), a, ph.x, ph.y);
                    } else if constexpr (PACKED) {
                        // fraction rounded to the nearest of its 2^fb steps, the last
                        // step kept below 1 so the entry still reads rows k0 and
                        // k0 + 1, the two samples the sum multiplies
                        return ((unsigned)rel << fb) | min(__float2uint_rn(a * frac_scale), frac_mask);
                    } else {
                        return make_float2(__int_as_float(base_row + rel), PRE ? wv * a : a);
                    }
                };
                if constexpr (DAS_BRICK_ALIGNED) {
                    float fv[NW], flv[NW];
                    bool okv[NW], any_v = false;
#pragma unroll
                    for (int i = 0; i < NW; ++i) {
                        fv[i] = tx[(v0 + i) * g.Q + q].x + dist[i];
                        flv[i] = floorf(fv[i]);
                        okv[i] = (flv[i] >= -1.f) && (flv[i] <= (float)(g.K - 1));
                        any_v |= okv[i];
                    }
                    const unsigned bal = __ballot_sync(0xffffffffu, any_v);
                    if (any_v) {
                        const int slot = __popc(bal & below);
                        // no term: rows K+1 and K+2 of this lane's slab (pad rows, zero)
                        const float pad = (float)g.K;
#pragma unroll
                        for (int i = 0; i < NW; ++i)
                            eb[i * ES + slot] = okv[i] ? make(fv[i], flv[i], tx[(v0 + i) * g.Q + q].y)
                                                    : make(pad, pad, 0.f);
                    }
                    n_mine = __popc(bal);
                } else {
#pragma unroll
                for (int i = 0; i < NW; ++i) {
                    const float f = tx[(v0 + i) * g.Q + q].x + dist[i];
                    const float fl = floorf(f);
                    // inside the aperture (dist < FAR) and a sample inside the
                    // record; false for NaN / inf
                    const bool ok = (fl >= -1.f) && (fl <= (float)(g.K - 1));
                    const unsigned bal = __ballot_sync(0xffffffffu, ok);
                    if (ok) eb[i * ES + __popc(bal & below)] = make(f, fl, tx[(v0 + i) * g.Q + q].y);
                    if (i == grp) n_mine = __popc(bal);
                }
                }
                __syncwarp();

                // ---- phase C: this group's list, U entries per trip, pipelined
                const float wq = tx[(v0 + grp) * g.Q + q].y;
                const float wqs = wq * frac_pow;               // (LOWF) wq 2^(23 - fb), exact
                const E *ev = eb + grp * ES;
                // first byte of this lane's chunk of the block's first row: packed
                // entries give a row relative to it
                const char *blk = permB + (long long)base_row * ROWB;
                // entry -> address of the lane's chunk of its first row, fraction
                // (and phase)
                auto decode = [&](E e, const char *&row, float &a, float2 &ph) {
                    if constexpr (!CPLX && PACKED) {
                        row = blk + (size_t)(e >> fb) * ROWB;
                        // the fraction bits as the mantissa of a float in [1, 2): in
                        // place as its low bits (LOWF: 1 + fraction 2^(fb - 23), the
                        // weight scaled to match), or shifted to its top (the row bits
                        // shift past the mantissa and are masked off)
                        if constexpr (LOWF) a = __int_as_float((e & frac_mask) | 0x3f800000u);
                        else a = __int_as_float(((e << frac_shift) & 0x007fffffu) | 0x3f800000u);
                        if constexpr (!FOLD) a -= 1.f;
                        ph = make_float2(1.f, 0.f);
                    } else {
                        row = permB + (long long)__float_as_int(e.x) * ROWB;
                        a = e.y;
                        if constexpr (CPLX) ph = make_float2(e.z, e.w);
                        else ph = make_float2(1.f, 0.f);
                    }
                };
                // the L 16-byte loads of one entry
                auto load_rows = [&](const char *p0, uint4 (&s)[L]) {
                    if constexpr (CONTIG) {
                        // chunks 2t, 2t + 1 of each row: s[2c + r] is chunk c of row r
                        load256(p0, s[0], s[2]);
                        load256(p0 + ROWB, s[1], s[3]);
                    } else if constexpr (SPLIT) {
                        s[0] = __ldg(reinterpret_cast<const uint4 *>(p0));
                    } else {
#pragma unroll
                        for (int c = 0; c < J; ++c) {
                            s[2 * c] = __ldg(reinterpret_cast<const uint4 *>(p0 + c * G * 16));
                            s[2 * c + 1] = __ldg(reinterpret_cast<const uint4 *>(p0 + ROWB + c * G * 16));
                        }
                    }
                };
                auto load_trip = [&](Trip<U, L> &tr, int i) {
                    E e[U];
                    if constexpr (!CPLX && PACKED && U % 2 == 0) {
                        // two 4-byte entries per 8-byte shared load
#pragma unroll
                        for (int u = 0; u < U; u += 2) {
                            const uint2 two = *reinterpret_cast<const uint2 *>(ev + i + u);
                            e[u] = two.x;
                            e[u + 1] = two.y;
                        }
                    } else if constexpr (!CPLX && !PACKED && U % 2 == 0) {
                        // two 8-byte entries per 16-byte shared load
#pragma unroll
                        for (int u = 0; u < U; u += 2) {
                            const float4 two = *reinterpret_cast<const float4 *>(ev + i + u);
                            e[u] = make_float2(two.x, two.y);
                            e[u + 1] = make_float2(two.z, two.w);
                        }
                    } else {
#pragma unroll
                        for (int u = 0; u < U; ++u) e[u] = ev[i + u];
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const char *row;
                        decode(e[u], row, tr.a[u], tr.ph[u]);
                        load_rows(row, tr.s[u]);
                    }
                };
                auto use_trip = [&](const Trip<U, L> &tr) {
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        accumulate<CPLX, HALF, SPLIT, WM, CS>(acc, wq, wqs, tr.a[u], tr.ph[u], tr.s[u], split_row);
                };
                int i = 0;
                if (n_mine >= U) {
                    Trip<U, L> ta, tb;
                    load_trip(ta, 0);
                    i = U;
                    for (;;) {
                        if (i + U > n_mine) { use_trip(ta); break; }
                        load_trip(tb, i);
                        i += U;
                        use_trip(ta);
                        if (i + U > n_mine) { use_trip(tb); break; }
                        load_trip(ta, i);
                        i += U;
                        use_trip(tb);
                    }
                }
                for (; i < n_mine; ++i) {
                    const char *row;
                    float a;
                    float2 ph;
                    uint4 s[L];
                    decode(ev[i], row, a, ph);
                    load_rows(row, s);
                    accumulate<CPLX, HALF, SPLIT, WM, CS>(acc, wq, wqs, a, ph, s, split_row);
                }
                // the next transmit writes the other buffer; the one after that
                // comes after the next __syncwarp
            }
        }
    }

    if constexpr (SPLIT) {
        // add the row-1 half of each chunk (held CPR lanes further on) to row 0
#pragma unroll
        for (int e = 0; e < NPA; ++e) {
            acc[0][e].x += __shfl_xor_sync(0xffffffffu, acc[0][e].x, CPR);
            acc[0][e].y += __shfl_xor_sync(0xffffffffu, acc[0][e].y, CPR);
        }
        if (split_row) return;
    }
    int n;
    if (!voxel(v0 + grp, n, nullptr)) return;
#pragma unroll
    for (int c = 0; c < NA; ++c)
#pragma unroll
        for (int e = 0; e < EPC; ++e) {
            const int chunk = SPLIT ? t : (CONTIG ? J * t + c : t + c * G);
            const long long idx = (long long)(chunk * EPC + e) * g.N + n;
            if constexpr (CPLX) {
                float2 *o = reinterpret_cast<float2 *>(out) + idx;
                const float2 v = CS
                                     ? make_float2(acc[c][e].x - acc[c][NPA - NP + e].y,
                                                   acc[c][e].y + acc[c][NPA - NP + e].x)
                                     : acc[c][e];
                *o = add_to_out ? make_float2(o->x + v.x, o->y + v.y) : v;
            } else {
                float *o = out + idx;
                const float v = (e & 1) ? acc[c][e >> 1].y : acc[c][e >> 1].x;
                *o = add_to_out ? *o + v : v;
            }
        }
}

template <int G, int J, bool CPLX, bool HALF, bool SPLIT, bool WIDE, int MWO = 0>
cudaError_t launch_one(const DasGeom &g, const RxPos *rx, const void *perm, const float *tau,
                       const float *w, void *out, cudaStream_t stream, int q0, int q1, int m0,
                       int m1, bool acc)
{
    constexpr int V = WARPS * (32 / G);
    constexpr int BX = BrickShape<V>::BX;
    constexpr int BY = V / BX;
    const int bricks_x = g.vox ? (g.N + V - 1) / V : (g.nx + BX - 1) / BX;
    const int bricks_y = g.vox ? 1 : (g.ny + BY - 1) / BY;
    const long long blocks = (long long)bricks_x * bricks_y * (g.vox ? 1 : g.nz);
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const size_t smem = smem_bytes<G, CPLX, HALF, WIDE>(g.Q);
    auto kernel = das_brick_kernel<G, J, CPLX, HALF, SPLIT, WIDE, MWO>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    // shared-memory share of the unified L1 / shared array the driver should
    // prefer: DAS_BRICK_CARVEOUT, or more where the CTAs the launch bounds ask
    // for need more (lists of float entries, long transmit tables)
    if (DAS_BRICK_CARVEOUT >= 0) {
        int dev = 0, per_sm = 0, reserved = 0;
        if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
        if ((err = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess)
            return err;
        if ((err = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess)
            return err;
        const double need = (double)min_blocks<G, J, CPLX, HALF, MWO>() * (double)(smem + reserved);
        int carveout = per_sm > 0 ? (int)std::ceil(100.0 * need / per_sm) : 100;
        if (carveout < DAS_BRICK_CARVEOUT) carveout = DAS_BRICK_CARVEOUT;
        if (carveout > 100) carveout = 100;
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, carveout);
        if (err != cudaSuccess) return err;
    }
    // CTAs resident at once: the SMs times the CTAs per SM the launch bounds ask for
    long long rot_wave = 0;
    if (DAS_BRICK_ROT > 0) {
        int dev = 0, sms = 0;
        if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
        if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
        rot_wave = (long long)sms * min_blocks<G, J, CPLX, HALF, MWO>() * DAS_BRICK_ROT / 100;
    }
    kernel<<<(int)blocks, THREADS, smem, stream>>>(g, rx, perm, tau, w, static_cast<float *>(out),
                                                   bricks_x, bricks_y, fraction_bits(g.K), q0, q1, m0, m1,
                                                   acc ? 1 : 0, rot_wave);
    return cudaGetLastError();
}

// Lanes per voxel G, chunks J, and split mode for B frames.
//   float32 / complex64 storage: pair mode, CPR = B * size / 16 chunks per row,
//     G = CPR if <= 8 (J = 1); rows of 16 or 32 chunks G = 16, J = CPR / 16
//     (16 lanes at one or two chunks each leave room for 32 warps per SM,
//     where 8 lanes at four chunks fit only 16); else G = 8, J = CPR / 8 in
//     {2, 4};
//   half / half2 storage: rows of <= 64 bytes (CPR <= 4) use split mode with
//     G = 2 CPR; wider rows pair mode with G = 8, J = CPR / 8 in {1, 2}.
bool choose(int B, bool cplx, bool half, int &G, int &J, bool &split)
{
    const int esz = half ? (cplx ? 4 : 2) : (cplx ? 8 : 4);
    if ((B * esz) % 16 != 0) return false;
    const int cpr = B * esz / 16;
    split = false;
    if (half) {
        if (cpr <= 4) {
            split = true;
            G = 2 * cpr;
            J = 1;
            return G == 2 || G == 4 || G == 8;
        }
        G = 8;
        J = cpr / 8;
        return cpr % 8 == 0 && (J == 1 || J == 2);
    }
    if (cpr == 8 && !cplx && DAS_BRICK_CONTIG_B32) {
        G = 4;          // 4 lanes x 8 frames, one 256-bit load per row and lane
        J = 2;
        return true;
    }
    if (cpr <= 8) {
        G = cpr;
        J = 1;
        return G == 2 || G == 4 || G == 8;
    }
    if (cpr == 16 || cpr == 32) {
        G = 16;         // rows of 256 or 512 bytes: 16 lanes, one or two chunks each
        J = cpr / 16;
        return true;
    }
    G = 8;
    J = cpr / 8;
    return cpr % 8 == 0 && (J == 2 || J == 4);
}

}  // namespace

bool brick_supported(int B, bool cplx, int K, bool half)
{
    int G, J;
    bool split;
    return K >= 2 && choose(B, cplx, half, G, J, split);
}

cudaError_t launch_brick(const DasGeom &g, const RxPos *rx, const void *perm, const float *tau,
                         const float *w, void *out, bool cplx, cudaStream_t stream, int q0, int q1,
                         bool accumulate, bool half, int m0, int m1)
{
    int G, J;
    bool split;
    if (q1 < 0) q1 = g.Q;
    if (m1 < 0) m1 = g.M;
    if (q0 < 0 || q0 > q1 || q1 > g.Q) return cudaErrorInvalidValue;
    // receiver ranges start on a block of MC receivers
    if (m0 < 0 || m0 > m1 || m1 > g.M || m0 % MC != 0) return cudaErrorInvalidValue;
    if (g.K < 2 || !choose(g.B, cplx, half, G, J, split)) return cudaErrorInvalidValue;
    // packed real entries while enough fraction bits remain, float entries beyond
    const bool wide = fraction_bits(g.K) < MIN_PACKED_BITS;
#define DAS_BRICK_ARGS g, rx, perm, tau, w, out, stream, q0, q1, m0, m1, accumulate
#define DAS_BRICK_CASE(GG, JJ, HH, SS)                                                         \
    if (G == GG && J == JJ && half == HH && split == SS)                                       \
        return cplx ? launch_one<GG, JJ, true, HH, SS, false>(DAS_BRICK_ARGS)                  \
                    : launch_one<GG, JJ, false, HH, SS, false>(DAS_BRICK_ARGS);
#define DAS_BRICK_CASE_WIDE(GG, JJ)                                                            \
    if (G == GG && J == JJ && !half && !split)                                                 \
        return cplx ? launch_one<GG, JJ, true, false, false, false>(DAS_BRICK_ARGS)            \
                    : (wide ? launch_one<GG, JJ, false, false, false, true>(DAS_BRICK_ARGS)    \
                            : launch_one<GG, JJ, false, false, false, false>(DAS_BRICK_ARGS));
    if (G == 4 && J == 1 && !cplx && !half && !split && !wide && DAS_BRICK_L2_WARPS_G4 > 0) {
        // the 4-lane float32 layout with more registers a warp when the padded
        // record fits in L2 (its loads then wait less and the extra registers
        // keep more of them in flight)
        int dev = 0, l2 = 0;
        cudaError_t err = cudaGetDevice(&dev);
        if (err == cudaSuccess) err = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
        if (err != cudaSuccess) return err;
        if ((double)g.B * g.Q * g.M * (g.K + 3) * sizeof(float) <= (double)l2)
            return launch_one<4, 1, false, false, false, false, DAS_BRICK_L2_WARPS_G4>(DAS_BRICK_ARGS);
    }
    DAS_BRICK_CASE_WIDE(2, 1) DAS_BRICK_CASE_WIDE(4, 1)
    DAS_BRICK_CASE_WIDE(8, 1) DAS_BRICK_CASE_WIDE(8, 2) DAS_BRICK_CASE_WIDE(4, 2)
    DAS_BRICK_CASE_WIDE(8, 4)
    DAS_BRICK_CASE_WIDE(16, 1) DAS_BRICK_CASE_WIDE(16, 2)
    DAS_BRICK_CASE(2, 1, true, true) DAS_BRICK_CASE(4, 1, true, true) DAS_BRICK_CASE(8, 1, true, true)
    DAS_BRICK_CASE(8, 1, true, false) DAS_BRICK_CASE(8, 2, true, false)
#undef DAS_BRICK_CASE
#undef DAS_BRICK_CASE_WIDE
#undef DAS_BRICK_ARGS
    return cudaErrorInvalidValue;
}

}  // namespace das
