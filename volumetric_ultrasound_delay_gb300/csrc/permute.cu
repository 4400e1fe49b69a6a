// RF layout permute: B x Q x M x K (k contiguous) -> a b-contiguous layout,
// as the batch-inner design needs (ffdas paper, Methods, batch-inner
// paragraph; ffdas docs, ALG2: the permute runs as part of the launch).
//
// For every (q, m) the (b, k) plane is transposed through shared memory in
// 32 x 32 element tiles, two tiles per block iteration so each thread keeps two
// 16-byte loads in flight.  Global loads read 16-byte vectors along k, global
// stores write 16-byte vectors along b; the shared tile has one element of
// padding per row, so the scalar shared-memory traffic is conflict-free for
// 4-byte elements.  The copy moves opaque element values and is bit-exact.
//
//   layout 0: out[((k*Q + q)*M + m)*B + b]         (K x Q x M x B)
//   layout 1: out[((q*M + m)*K + k)*B + b]         (Q x M x K x B)
//   layout 2: out[((q*M + m)*(K+3) + k + 1)*B + b] (Q x M x (K+3) x B: every
//             (q, m) slab has a row before k = 0 and two rows after k = K-1
//             that this kernel never writes; the brick kernel keeps them zero)
//   layout 3: out[(((k+1)*Q + q)*M + m)*B + b]     ((K+2) x Q x M x B: the
//             batch-inner layout with a plane before k = 0 and one after
//             k = K-1 that this kernel never writes; the BI kernel keeps them
//             zero)
//
// With half-precision storage the copy converts float32 -> half and complex64
// -> half2 (round to nearest) as it writes: the pages' FP16 variants fuse that
// conversion into the permute (ffdas paper, Methods, FP16 paragraphs).
//
// On request the copy also reports whether the record holds a non-finite
// float32 value (NaN or inf, any component): it sets *nonfinite to 1, which
// the caller clears beforehand.  The pair kernel reads that flag to decide
// whether zero weights may multiply samples (see das_pair.cu).
#include <cuda_fp16.h>

#include <cstdint>
#include <cstring>

#include "das_internal.cuh"

namespace das {
namespace {

constexpr int TILE = 32;
constexpr int THREADS = 256;

// tiles along k per block iteration: 4 for 4-byte elements (0.74 ms for the
// 2.4 GB float32 record of the 32 x 32-array volume, against 0.84 ms with 2),
// 2 for 8-byte ones (4 would double the shared tile and cost 40 %)
template <typename T>
constexpr int sub_tiles() { return sizeof(T) >= 8 ? 2 : 4; }

// element conversion on the way out: identity, or float -> half / float2 -> half2
// (round to nearest) for half-precision storage of the copy
template <typename TO, typename TI>
__device__ __forceinline__ TO convert(TI v) { return v; }

// 1 if a 32-bit word is a float32 NaN or inf
__device__ __forceinline__ unsigned not_finite(unsigned w) { return (w & 0x7f800000u) == 0x7f800000u; }
template <>
__device__ __forceinline__ __half convert<__half, float>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __half2 convert<__half2, float2>(float2 v) { return __float22half2_rn(v); }

// CHECK: also report non-finite float32 values (4- and 8-byte elements)
template <typename T, typename TO, bool CHECK>
__global__ void __launch_bounds__(THREADS)
permute_kernel(const T *__restrict__ in, TO *__restrict__ out, int B, int QM, int K,
               long long osk, long long osqm, long long n_blocks, int blocks_b, int blocks_k,
               int vec_in, int vec_out, int qm0, unsigned *__restrict__ nonfinite)
{
    static_assert(!CHECK || sizeof(T) % 4 == 0, "only float data is checked");
    unsigned bad = 0u;
    constexpr int V = 16 / sizeof(T);            // input elements per 16-byte vector
    constexpr int VPR = TILE / V;                // input vectors per 32-element row
    constexpr int VO = 16 / sizeof(TO);          // output elements per 16-byte vector
    constexpr int VPRO = TILE / VO;              // output vectors per 32-element row
    constexpr int SUB = sub_tiles<T>();
    __shared__ T tile[SUB][TILE][TILE + 1];
    const int tid = threadIdx.x;

    for (long long t = blockIdx.x; t < n_blocks; t += gridDim.x) {
        const int tk = (int)(t % blocks_k);
        const long long r = t / blocks_k;
        const int tb = (int)(r % blocks_b);
        const int qm = qm0 + (int)(r / blocks_b);
        const int b0 = tb * TILE;
        const int k0 = tk * TILE * SUB;

        // ---- load SUB tiles of 32 (b) x 32 (k)
        if (vec_in) {
#pragma unroll
            for (int s = 0; s < SUB; ++s) {
                for (int i = tid; i < TILE * VPR; i += THREADS) {
                    const int row = i / VPR, v = i % VPR;
                    const int b = b0 + row, k = k0 + s * TILE + v * V;
                    if (b < B && k < K) {   // K % V == 0, so the whole vector is inside
                        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(
                            in + ((long long)b * QM + qm) * K + k));
                        if constexpr (CHECK)
                            bad |= not_finite(u.x) | not_finite(u.y) | not_finite(u.z) | not_finite(u.w);
                        T vals[V];
                        memcpy(vals, &u, sizeof(u));
#pragma unroll
                        for (int j = 0; j < V; ++j) tile[s][row][v * V + j] = vals[j];
                    }
                }
            }
        } else {
            for (int s = 0; s < SUB; ++s)
                for (int i = tid; i < TILE * TILE; i += THREADS) {
                    const int row = i / TILE, kk = i % TILE;
                    const int b = b0 + row, k = k0 + s * TILE + kk;
                    if (b < B && k < K) {
                        const T v = in[((long long)b * QM + qm) * K + k];
                        if constexpr (CHECK) {
                            unsigned w[sizeof(T) / 4];
                            memcpy(w, &v, sizeof(T));
#pragma unroll
                            for (int j = 0; j < (int)(sizeof(T) / 4); ++j) bad |= not_finite(w[j]);
                        }
                        tile[s][row][kk] = v;
                    }
                }
        }
        __syncthreads();

        // ---- store: rows of k, b contiguous
        if (vec_out) {
#pragma unroll
            for (int s = 0; s < SUB; ++s) {
                for (int i = tid; i < TILE * VPRO; i += THREADS) {
                    const int krow = i / VPRO, v = i % VPRO;
                    const int k = k0 + s * TILE + krow, b = b0 + v * VO;
                    if (k < K && b < B) {   // B % VO == 0
                        TO vals[VO];
#pragma unroll
                        for (int j = 0; j < VO; ++j) vals[j] = convert<TO>(tile[s][v * VO + j][krow]);
                        uint4 u;
                        memcpy(&u, vals, sizeof(u));
                        *reinterpret_cast<uint4 *>(out + (long long)k * osk + (long long)qm * osqm + b) = u;
                    }
                }
            }
        } else {
            for (int s = 0; s < SUB; ++s)
                for (int i = tid; i < TILE * TILE; i += THREADS) {
                    const int krow = i / TILE, bb = i % TILE;
                    const int k = k0 + s * TILE + krow, b = b0 + bb;
                    if (k < K && b < B)
                        out[(long long)k * osk + (long long)qm * osqm + b] = convert<TO>(tile[s][bb][krow]);
                }
        }
        __syncthreads();
    }
    if constexpr (CHECK) {
        const unsigned any = __ballot_sync(0xffffffffu, bad != 0u);
        if (any != 0u && (threadIdx.x & 31) == __ffs(any) - 1) atomicOr(nonfinite, 1u);
    }
}

template <typename T, typename TO = T>
cudaError_t launch_typed(const void *in, void *out, int B, int Q, int M, int K, int layout,
                         int num_sms, cudaStream_t stream, int q0, int q1, unsigned *nonfinite)
{
    constexpr int V = 16 / sizeof(T);
    constexpr int VO = 16 / sizeof(TO);
    const int QM = Q * M;
    const bool kmajor = layout == 0 || layout == 3;
    const long long osk = kmajor ? (long long)QM * B : (long long)B;
    const long long osqm = kmajor ? (long long)B
                         : layout == 1 ? (long long)K * B : (long long)(K + 3) * B;
    if (layout == 2) out = static_cast<TO *>(out) + B;                      // row k = 0 of slab 0
    if (layout == 3) out = static_cast<TO *>(out) + (long long)QM * B;      // plane k = 0
    const int blocks_b = (B + TILE - 1) / TILE;
    constexpr int SUB = sub_tiles<T>();
    const int blocks_k = (K + TILE * SUB - 1) / (TILE * SUB);
    const long long n_blocks = (long long)(q1 - q0) * M * blocks_b * blocks_k;
    if (n_blocks == 0) return cudaSuccess;
    const bool in_al = (reinterpret_cast<uintptr_t>(in) % 16) == 0;
    const bool out_al = (reinterpret_cast<uintptr_t>(out) % 16) == 0;
    const int vec_in = in_al && (K % V == 0);
    const int vec_out = out_al && (B % VO == 0) && (osk % VO == 0) && (osqm % VO == 0);
    const long long cap = (long long)num_sms * 8;
    const int grid = (int)(n_blocks < cap ? n_blocks : cap);
    if constexpr (sizeof(T) % 4 == 0) {
        if (nonfinite) {
            permute_kernel<T, TO, true><<<grid, THREADS, 0, stream>>>(
                static_cast<const T *>(in), static_cast<TO *>(out), B, QM, K, osk, osqm, n_blocks,
                blocks_b, blocks_k, vec_in, vec_out, q0 * M, nonfinite);
            return cudaGetLastError();
        }
    }
    permute_kernel<T, TO, false><<<grid, THREADS, 0, stream>>>(
        static_cast<const T *>(in), static_cast<TO *>(out), B, QM, K, osk, osqm, n_blocks,
        blocks_b, blocks_k, vec_in, vec_out, q0 * M, nullptr);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_permute(const void *in, void *out, int elem_bytes, int B, int Q, int M, int K,
                           int layout, int num_sms, cudaStream_t stream, int q0, int q1,
                           bool to_half, unsigned *nonfinite)
{
    if (q1 < 0) q1 = Q;
    if (q0 < 0 || q0 > q1 || q1 > Q) return cudaErrorInvalidValue;
    if (to_half) {
        switch (elem_bytes) {
        case 4: return launch_typed<float, __half>(in, out, B, Q, M, K, layout, num_sms, stream, q0, q1, nonfinite);
        case 8: return launch_typed<float2, __half2>(in, out, B, Q, M, K, layout, num_sms, stream, q0, q1, nonfinite);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (elem_bytes) {
    case 2: return launch_typed<unsigned short>(in, out, B, Q, M, K, layout, num_sms, stream, q0, q1, nonfinite);
    case 4: return launch_typed<float>(in, out, B, Q, M, K, layout, num_sms, stream, q0, q1, nonfinite);
    case 8: return launch_typed<float2>(in, out, B, Q, M, K, layout, num_sms, stream, q0, q1, nonfinite);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace das
