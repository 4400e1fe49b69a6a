// C ABI of libdas: plan management, argument checks and kernel dispatch.
// Every entry point validates on the host, launches nothing when it rejects a
// call, and maps CUDA failures to DAS_ERR_CUDA with a readable message.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "das_internal.cuh"

namespace {

thread_local char g_err[512] = "";

das_status fail(das_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

das_status cuda_fail(cudaError_t e, const char *what)
{
    if (e == cudaErrorMemoryAllocation)
        return fail(DAS_ERR_OUT_OF_MEMORY, "%s: %s", what, cudaGetErrorString(e));
    return fail(DAS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

void das::record_error(const char *msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }

struct das_plan_s {
    das_grid grid{};
    float c = 0, fs = 0, t0 = 0, fnum = 0;
    das_dtype dtype = DAS_F32;
    int B = 0, Q = 0, M = 0, K = 0;
    long long N = 0;
    int device = 0;
    int num_sms = 1;
    int kernel = DAS_KERNEL_AUTO;
    int bi_group = 0;
    double f_demod = 0.0;
    int timing = 0;
    bool timed_once = false;
    bool last_had_permute = false;
    cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
    // the plan's own stream (allocations, uploads, stream-ordered frees) and the
    // event recorded after the last work each call queued on the caller's stream
    cudaStream_t own = nullptr;
    cudaEvent_t done = nullptr;
    bool used = false;
    RxPos *d_rx = nullptr;
    float4 *d_vox = nullptr;                  // voxel list (sample units, slot order), list plans only
    int *d_order = nullptr;                   // list plans: caller's index of each slot
    Pos64 *d_rx64 = nullptr, *d_vox64 = nullptr;   // double copies, float64 / complex128 plans
    void *d_perm = nullptr;
    unsigned *d_flag = nullptr;               // set by the permute when the record holds NaN / inf
    size_t perm_bytes = 0;
    int perm_zero_layout = -1;     // padded layout (2 or 3) whose pad rows the scratch holds as zeros
    // device staging of das_beamform_host, and its copy stream / events
    void *d_rf = nullptr, *d_out = nullptr;
    float *d_tau = nullptr, *d_w = nullptr;
    int host_groups = 0;                      // DAS_OPT_HOST_GROUPS (0 = automatic)
    int rx_groups = 1;                        // DAS_OPT_RX_GROUPS (0 = automatic)
    int tx_groups = 0;                        // DAS_OPT_TX_GROUPS (0 = automatic)
    int storage = DAS_STORAGE_NATIVE;         // DAS_OPT_STORAGE
    cudaStream_t copy_stream = nullptr;
    std::vector<cudaEvent_t> copy_ev;         // [0]: start, [1]: tau/w copied, [2+g]: group g copied
    std::vector<cudaEvent_t> used_ev;         // [g]: the staging copy of group g read (volume streams)
    DasGeom geom{};
    DasGeom64 geom64{};

    bool is_double() const { return dtype == DAS_F64 || dtype == DAS_C128; }
    bool is_complex() const { return dtype == DAS_C64 || dtype == DAS_C128 || dtype == DAS_C32H; }
    // single-precision complex: complex64 or half2 samples, complex64 output
    bool cplx32() const { return dtype == DAS_C64 || dtype == DAS_C32H; }
    // the record arrives in half precision (DAS_F16, DAS_C32H)
    bool half_in() const { return dtype == DAS_F16 || dtype == DAS_C32H; }
    // the kernels read half-precision rows: half input, or float input stored as half
    bool half_rows() const { return half_in() || storage == DAS_STORAGE_F16; }
    // the permute rounds float32 / complex64 samples to half precision
    bool convert_half() const { return !half_in() && storage == DAS_STORAGE_F16; }
    // bytes of one record element as the caller passes it
    size_t elem_bytes() const
    {
        switch (dtype) {
        case DAS_F16: return 2;
        case DAS_F32: case DAS_C32H: return 4;
        case DAS_C128: return 16;
        default: return 8;
        }
    }
    // bytes of one element of the permuted copy the kernels read
    size_t row_elem_bytes() const { return convert_half() ? elem_bytes() / 2 : elem_bytes(); }
    // bytes of one output element (float32 / complex64 for the half inputs)
    size_t out_elem_bytes() const { return dtype == DAS_F16 ? 4 : (dtype == DAS_C32H ? 8 : elem_bytes()); }
    size_t rf_bytes() const { return (size_t)B * Q * M * K * elem_bytes(); }
    size_t padded_bytes() const { return (size_t)B * Q * M * (K + 3) * elem_bytes(); }
    size_t out_bytes() const { return (size_t)B * (size_t)N * out_elem_bytes(); }
    size_t txw_bytes() const { return (size_t)Q * (size_t)N * sizeof(float); }
};

namespace {

int resolve_kernel(const das_plan_s *p)
{
    const bool cplx = p->cplx32();
    if (p->kernel != DAS_KERNEL_AUTO) return p->kernel;
    if (p->is_double()) return DAS_KERNEL_BL;                     // the only double-precision kernel
    if (p->half_rows()) return DAS_KERNEL_BRICK;                  // half rows: brick (or BI on request)
    if (das::brick_supported(p->B, cplx, p->K)) return DAS_KERNEL_BRICK;
    if (p->K >= 2 && das::bi_supported(p->B, cplx, p->bi_group, p->Q, p->M, p->K)) return DAS_KERNEL_BI;
    return DAS_KERNEL_BL;
}

// Order in which a voxel list plan keeps its voxels: deepest first in depth
// bands, then along a 2-D Morton curve in x-y, on cells of the list's mean
// spacing.  Neighbouring slots are then neighbours in space, as the bricks of
// a grid are (same rows of the record, warm caches), whatever order the
// caller lists them in.  Returns an empty vector when the points span no
// volume worth ordering (then slot = index).
std::vector<int> compact_order(const float *xyz, int N)
{
    std::vector<int> order;
    if (N < 2) return order;
    double lo[3] = {xyz[0], xyz[1], xyz[2]}, hi[3] = {xyz[0], xyz[1], xyz[2]};
    for (int n = 1; n < N; ++n)
        for (int d = 0; d < 3; ++d) {
            lo[d] = std::min(lo[d], (double)xyz[3 * n + d]);
            hi[d] = std::max(hi[d], (double)xyz[3 * n + d]);
        }
    // mean spacing: the cube root of the volume per point, over the extents
    // that are not flat
    double vol = 1.0;
    int dims = 0;
    for (int d = 0; d < 3; ++d)
        if (hi[d] > lo[d]) { vol *= hi[d] - lo[d]; ++dims; }
    if (dims == 0) return order;
    const double h = std::pow(vol / N, 1.0 / dims);
    if (!(h > 0.0) || !std::isfinite(h)) return order;
    auto cell = [&](double v, double origin) -> uint32_t {
        const double c = std::floor((v - origin) / h);
        return c <= 0.0 ? 0u : (c >= 65535.0 ? 65535u : (uint32_t)c);
    };
    auto spread = [](uint32_t v) -> uint64_t {   // bit i of v to bit 2i
        uint64_t x = v & 0xffffu;
        x = (x | (x << 8)) & 0x00ff00ffull;
        x = (x | (x << 4)) & 0x0f0f0f0full;
        x = (x | (x << 2)) & 0x33333333ull;
        x = (x | (x << 1)) & 0x55555555ull;
        return x;
    };
    std::vector<uint64_t> key(N);
    for (int n = 0; n < N; ++n) {
        const uint64_t band = cell(hi[2] - (double)xyz[3 * n + 2], 0.0);   // 0 = deepest
        key[n] = (band << 32) | (spread(cell(xyz[3 * n], lo[0])) |
                                 (spread(cell(xyz[3 * n + 1], lo[1])) << 1));
    }
    order.resize(N);
    for (int n = 0; n < N; ++n) order[n] = n;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return key[a] < key[b]; });
    return order;
}

// Receiver groups of the brick kernel when DAS_OPT_RX_GROUPS is 0: enough that
// one group's share of the permuted record fits in half of the L2.
int auto_rx_groups(const das_plan_s *p)
{
    int l2 = 0, dev = p->device;
    if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess || l2 <= 0) {
        cudaGetLastError();
        return 1;
    }
    const size_t elem = p->row_elem_bytes();
    const size_t bytes = (size_t)p->B * p->Q * p->M * (p->K + 3) * elem;
    const size_t share = (size_t)l2 / 2;
    const size_t R = (bytes + share - 1) / share;
    return R < 1 ? 1 : (R > 64 ? 64 : (int)R);
}

// Transmit groups of the brick kernel when DAS_OPT_TX_GROUPS is 0: enough that
// one group's share of the permuted record is at most 16 times the L2.  The
// CTAs resident at one time read a few hundred rows of every slab of their
// group's transmits; with a share of that size those rows stay in L2 until the
// neighbouring bricks that read them again have done so.  Each extra launch
// repeats the receive distances, so the split is made only where the record's
// re-reads weigh against the work: at least one byte of record per 64
// accumulations (B N Q M); below that the kernel spends so long on each byte it
// reads that DRAM re-reads cost nothing.
int auto_tx_groups(const das_plan_s *p)
{
    int l2 = 0;
    if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, p->device) != cudaSuccess || l2 <= 0) {
        cudaGetLastError();
        return 1;
    }
    const size_t elem = p->row_elem_bytes();
    const size_t bytes = (size_t)p->B * p->Q * p->M * (p->K + 3) * elem;
    const double accumulations = (double)p->B * (double)p->N * (double)p->Q * (double)p->M;
    if ((double)bytes * 64.0 < accumulations) return 1;
    const size_t share = (size_t)16 * (size_t)l2;
    const size_t T = (bytes + share - 1) / share;
    return T < 1 ? 1 : (T > (size_t)p->Q ? p->Q : (int)T);
}

// launches of the brick kernel in one das_beamform: receiver groups x transmit groups
void brick_groups(const das_plan_s *p, int &R, int &T)
{
    const int blocks = (p->M + 31) / 32;
    R = p->rx_groups > 0 ? p->rx_groups : auto_rx_groups(p);
    if (R > blocks) R = blocks;
    T = p->tx_groups > 0 ? p->tx_groups : auto_tx_groups(p);
    if (T > p->Q) T = p->Q;
}

das_status check_supported(const das_plan_s *p, int kernel)
{
    const bool cplx = p->cplx32();
    const bool half = p->half_rows();
    if (half && kernel != DAS_KERNEL_BRICK && kernel != DAS_KERNEL_BI)
        return fail(DAS_ERR_UNSUPPORTED,
                    "half-precision records and storage are served by the brick and BI kernels only");
    if (p->is_double() && kernel != DAS_KERNEL_BL)
        return fail(DAS_ERR_UNSUPPORTED, "float64 / complex128 plans are served by the BL kernel only");
    switch (kernel) {
    case DAS_KERNEL_BL: return DAS_OK;
    case DAS_KERNEL_BI:
        if (p->K < 2 || !das::bi_supported(p->B, cplx, p->bi_group, p->Q, p->M, p->K, half))
            return fail(DAS_ERR_UNSUPPORTED,
                        "BI kernel needs K >= 2, B a multiple of the group's 16-byte chunks "
                        "(half storage: one chunk per lane), its transmit table in shared memory "
                        "and a record of < 2^32 16-byte chunks (B=%d, group=%d, Q=%d)",
                        p->B, p->bi_group, p->Q);
        return DAS_OK;
    case DAS_KERNEL_BRICK:
        if (!das::brick_supported(p->B, cplx, p->K, half))
            return fail(DAS_ERR_UNSUPPORTED,
                        "brick kernel needs K >= 2 and B * element size in {32, 64, 128, 256, 512} "
                        "bytes (half storage: {16, ..., 64, 128, 256}) (B=%d)", p->B);
        return DAS_OK;
    case DAS_KERNEL_PAIR:
        if (!das::pair_supported(p->B, cplx, p->K))
            return fail(DAS_ERR_UNSUPPORTED,
                        "pair kernel needs a float32 record with B in {16, 32, 64} and K >= 2 (B=%d)",
                        p->B);
        if (das::pair_smem_bytes(p->B, p->Q) > 227 * 1024)
            return fail(DAS_ERR_UNSUPPORTED, "pair kernel: transmit table of Q=%d does not fit shared memory",
                        p->Q);
        return DAS_OK;
    case DAS_KERNEL_WINDOW:
        if (!das::window_supported(p->B, cplx, p->K, p->Q, p->M))
            return fail(DAS_ERR_UNSUPPORTED,
                        "window kernel needs a float32 record with B in {8, 16, 32}, K >= 2, "
                        "Q x M x (K+3) < 2^31 and its transmit table in shared memory "
                        "(B=%d, Q=%d)", p->B, p->Q);
        return DAS_OK;
    default: return fail(DAS_ERR_INVALID_ARG, "unknown kernel %d", kernel);
    }
}

// Device memory of a plan comes from the stream-ordered allocator on the
// plan's own stream; once these return it is ready for use on any stream.
template <typename T>
cudaError_t plan_alloc(das_plan_s *p, T **ptr, size_t bytes)
{
    void *v = nullptr;
    cudaError_t e = cudaMallocAsync(&v, bytes, p->own);
    if (e == cudaSuccess) e = cudaStreamSynchronize(p->own);
    if (e != cudaSuccess) {
        if (v) cudaFreeAsync(v, p->own);
        v = nullptr;
        cudaGetLastError();
    }
    *ptr = static_cast<T *>(v);
    return e;
}

template <typename T>
cudaError_t plan_upload(das_plan_s *p, T **ptr, const void *src, size_t bytes)
{
    cudaError_t e = plan_alloc(p, ptr, bytes);
    if (e == cudaSuccess) e = cudaMemcpyAsync(*ptr, src, bytes, cudaMemcpyHostToDevice, p->own);
    if (e == cudaSuccess) e = cudaStreamSynchronize(p->own);
    return e;
}

// Releases everything the plan owns without waiting on the host: the device
// buffers are freed on the plan's own stream after the event that marks the
// end of the plan's last queued work, so neither this plan's queued work nor
// any other stream is waited for; events and streams with work still pending
// are released by CUDA once that work completes.
void release(das_plan_s *p)
{
    if (p->own) {
        void *bufs[] = {p->d_rx, p->d_vox, p->d_order, p->d_rx64, p->d_vox64,
                        p->d_perm, p->d_flag, p->d_rf, p->d_out, p->d_tau, p->d_w};
        if (p->used && p->done) cudaStreamWaitEvent(p->own, p->done, 0);
        for (void *b : bufs)
            if (b) cudaFreeAsync(b, p->own);
    }
    for (auto &e : p->ev)
        if (e) cudaEventDestroy(e);
    for (auto &e : p->copy_ev)
        if (e) cudaEventDestroy(e);
    for (auto &e : p->used_ev)
        if (e) cudaEventDestroy(e);
    if (p->done) cudaEventDestroy(p->done);
    if (p->copy_stream) cudaStreamDestroy(p->copy_stream);
    if (p->own) cudaStreamDestroy(p->own);
    cudaGetLastError();
}

// Records the plan's done event on the caller's stream when a call returns,
// by whatever path, after it may have queued work there.
struct DoneMark {
    das_plan_s *p;
    cudaStream_t stream;
    ~DoneMark()
    {
        if (cudaEventRecord(p->done, stream) == cudaSuccess) p->used = true;
        else cudaGetLastError();
    }
};

// Allocates the permute scratch on first use (sized for the brick kernel's
// padded layout, the larger one) and zeroes it when a padded layout is about
// to be used after
// the scratch held something else; the permute never writes the pad rows.
das_status ensure_scratch(das_plan_s *p, int layout, cudaStream_t stream)
{
    if (!p->d_flag) {
        cudaError_t e = plan_alloc(p, &p->d_flag, 256);
        if (e != cudaSuccess) return cuda_fail(e, "flag allocation");
    }
    if (!p->d_perm) {
        cudaError_t e = plan_alloc(p, &p->d_perm, p->padded_bytes());
        if (e != cudaSuccess) return cuda_fail(e, "permute scratch allocation");
        p->perm_bytes = p->padded_bytes();
        p->perm_zero_layout = -1;
    }
    if (p->perm_zero_layout != layout) {
        cudaError_t e = cudaMemsetAsync(p->d_perm, 0, p->padded_bytes(), stream);
        if (e != cudaSuccess) return cuda_fail(e, "zeroing the permute scratch");
        p->perm_zero_layout = layout;
    }
    return DAS_OK;
}

// Restores the caller's current device on scope exit.
struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) cudaSetDevice(dev);
        else prev = -1;
    }
    ~DeviceGuard()
    {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

}  // namespace

extern "C" {

const char *das_last_error_string(void) { return g_err; }

const char *das_version(void) { return "1.0.0"; }

das_status das_plan_create(das_plan *plan, const das_grid *grid, const float *rx_xyz, float c,
                           float fs, float t0, float fnum, das_dtype dtype, int B, int Q, int M,
                           int K)
{
    g_err[0] = '\0';
    if (!plan) return fail(DAS_ERR_INVALID_ARG, "plan is NULL");
    *plan = nullptr;
    if (!grid) return fail(DAS_ERR_INVALID_ARG, "grid is NULL");
    if (!rx_xyz) return fail(DAS_ERR_INVALID_ARG, "rx_xyz is NULL");
    if (grid->nx < 1 || grid->ny < 1 || grid->nz < 1)
        return fail(DAS_ERR_INVALID_ARG, "grid dimensions must be >= 1");
    if (grid->xyz) {
        const long long n = (long long)grid->nx * grid->ny * grid->nz;
        if (n >= (1LL << 31)) return fail(DAS_ERR_INVALID_ARG, "nx*ny*nz must be < 2^31");
        return das_plan_create_points(plan, grid->xyz, (int)n, rx_xyz, c, fs, t0, fnum, dtype, B, Q,
                                      M, K);
    }
    const float gf[6] = {grid->x0, grid->y0, grid->z0, grid->dx, grid->dy, grid->dz};
    for (float v : gf)
        if (!std::isfinite(v)) return fail(DAS_ERR_INVALID_ARG, "grid origin/spacing not finite");
    if (!(c > 0.f) || !std::isfinite(c)) return fail(DAS_ERR_INVALID_ARG, "c must be > 0");
    if (!(fs > 0.f) || !std::isfinite(fs)) return fail(DAS_ERR_INVALID_ARG, "fs must be > 0");
    if (!std::isfinite(t0) || !std::isfinite(fnum))
        return fail(DAS_ERR_INVALID_ARG, "t0 and fnum must be finite");
    if (dtype < DAS_F32 || dtype > DAS_C32H) return fail(DAS_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (B < 1 || Q < 1 || M < 1 || K < 1) return fail(DAS_ERR_INVALID_ARG, "B, Q, M, K must be >= 1");
    const long long N = (long long)grid->nx * grid->ny * grid->nz;
    if ((long long)Q * M * (K + 3) >= (1LL << 31))
        return fail(DAS_ERR_INVALID_ARG, "Q*M*(K+3) must be < 2^31");
    if (N * B >= (1LL << 31)) return fail(DAS_ERR_INVALID_ARG, "B*N must be < 2^31");
    if ((long long)Q * N >= (1LL << 40)) return fail(DAS_ERR_INVALID_ARG, "Q*N too large");
    if (K >= (1 << 22)) return fail(DAS_ERR_INVALID_ARG, "K must be < 2^22");
    for (int i = 0; i < 3 * M; ++i)
        if (!std::isfinite(rx_xyz[i])) return fail(DAS_ERR_INVALID_ARG, "receiver position not finite");

    das_plan_s *p = new (std::nothrow) das_plan_s;
    if (!p) return fail(DAS_ERR_OUT_OF_MEMORY, "host allocation of the plan failed");
    p->grid = *grid;
    p->grid.xyz = nullptr;   // the caller's list is copied below, not kept
    p->c = c; p->fs = fs; p->t0 = t0; p->fnum = fnum;
    p->dtype = dtype;
    p->B = B; p->Q = Q; p->M = M; p->K = K;
    p->N = N;
    cudaError_t e = cudaGetDevice(&p->device);
    if (e != cudaSuccess) { delete p; return cuda_fail(e, "cudaGetDevice"); }
    e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
    if (e != cudaSuccess) { delete p; return cuda_fail(e, "cudaDeviceGetAttribute"); }
    e = cudaStreamCreateWithFlags(&p->own, cudaStreamNonBlocking);
    if (e != cudaSuccess) { p->own = nullptr; delete p; return cuda_fail(e, "plan stream"); }
    e = cudaEventCreateWithFlags(&p->done, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        p->done = nullptr;
        release(p);
        delete p;
        return cuda_fail(e, "plan event");
    }

    // positions in sample units (metres * fs / c), scaled in double
    const double s = (double)fs / (double)c;
    std::vector<RxPos> hrx(M);
    for (int m = 0; m < M; ++m)
        hrx[m] = make_float4((float)(rx_xyz[3 * m] * s), (float)(rx_xyz[3 * m + 1] * s),
                             (float)(rx_xyz[3 * m + 2] * s), 0.f);
    DasGeom &g = p->geom;
    g.nx = grid->nx; g.ny = grid->ny; g.nz = grid->nz; g.N = (int)N;
    g.x0 = (float)(grid->x0 * s); g.y0 = (float)(grid->y0 * s); g.z0 = (float)(grid->z0 * s);
    g.dx = (float)(grid->dx * s); g.dy = (float)(grid->dy * s); g.dz = (float)(grid->dz * s);
    g.fs = fs;
    g.t0fs = (float)((double)t0 * fs);
    g.aperture = fnum > 0.f;
    g.ap2 = g.aperture ? (float)(4.0 * (double)fnum * fnum) : 0.f;
    g.fd_over_fs = 0.f;
    g.rotate = 0;
    g.B = B; g.Q = Q; g.M = M; g.K = K;

    DasGeom64 &g64 = p->geom64;
    g64.nx = g.nx; g64.ny = g.ny; g64.nz = g.nz; g64.N = g.N;
    g64.x0 = grid->x0 * s; g64.y0 = grid->y0 * s; g64.z0 = grid->z0 * s;
    g64.dx = grid->dx * s; g64.dy = grid->dy * s; g64.dz = grid->dz * s;
    g64.fs = fs;
    g64.t0fs = (double)t0 * fs;
    g64.aperture = g.aperture;
    g64.ap2 = g.aperture ? 4.0 * (double)fnum * fnum : 0.0;
    g64.fd_over_fs = 0.0;
    g64.B = B; g64.Q = Q; g64.M = M; g64.K = K;
    g64.vox = nullptr;

    e = plan_upload(p, &p->d_rx, hrx.data(), sizeof(RxPos) * M);
    if (e == cudaSuccess && p->is_double()) {
        std::vector<Pos64> h64(M);
        for (int m = 0; m < M; ++m)
            h64[m] = Pos64{rx_xyz[3 * m] * s, rx_xyz[3 * m + 1] * s, rx_xyz[3 * m + 2] * s, 0.0};
        e = plan_upload(p, &p->d_rx64, h64.data(), sizeof(Pos64) * M);
    }
    if (e != cudaSuccess) {
        release(p);
        delete p;
        return cuda_fail(e, "receiver upload");
    }
    *plan = p;
    return DAS_OK;
}

das_status das_plan_create_points(das_plan *plan, const float *voxel_xyz, int N,
                                  const float *rx_xyz, float c, float fs, float t0, float fnum,
                                  das_dtype dtype, int B, int Q, int M, int K)
{
    g_err[0] = '\0';
    if (!plan) return fail(DAS_ERR_INVALID_ARG, "plan is NULL");
    *plan = nullptr;
    if (!voxel_xyz) return fail(DAS_ERR_INVALID_ARG, "voxel_xyz is NULL");
    if (N < 1) return fail(DAS_ERR_INVALID_ARG, "N must be >= 1");
    if (!(c > 0.f) || !(fs > 0.f) || !std::isfinite(c) || !std::isfinite(fs))
        return fail(DAS_ERR_INVALID_ARG, "c and fs must be > 0");
    for (long long i = 0; i < 3LL * N; ++i)
        if (!std::isfinite(voxel_xyz[i])) return fail(DAS_ERR_INVALID_ARG, "voxel position not finite");
    // a 1 x 1 x N grid carries the sizes; the positions come from the list
    const das_grid grid = {1, 1, N, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, nullptr};
    das_status st = das_plan_create(plan, &grid, rx_xyz, c, fs, t0, fnum, dtype, B, Q, M, K);
    if (st != DAS_OK) return st;
    das_plan_s *p = *plan;
    const double s = (double)fs / (double)c;
    // slot k holds voxel order[k]; positions are uploaded in slot order
    const std::vector<int> order = compact_order(voxel_xyz, N);
    auto index = [&](int k) { return order.empty() ? k : order[k]; };
    std::vector<float4> hv(N);
    for (int k = 0; k < N; ++k) {
        const float *v = voxel_xyz + 3 * (size_t)index(k);
        hv[k] = make_float4((float)(v[0] * s), (float)(v[1] * s), (float)(v[2] * s), 0.f);
    }
    cudaError_t e;
    {
        DeviceGuard dg(p->device);
        e = plan_upload(p, &p->d_vox, hv.data(), sizeof(float4) * (size_t)N);
        if (e == cudaSuccess && !order.empty())
            e = plan_upload(p, &p->d_order, order.data(), sizeof(int) * (size_t)N);
    }
    if (e != cudaSuccess) {
        das_plan_destroy(p);
        *plan = nullptr;
        cudaGetLastError();
        return cuda_fail(e, "voxel list upload");
    }
    p->geom.vox = p->d_vox;
    p->geom.order = p->d_order;
    p->geom64.order = p->d_order;
    if (p->is_double()) {
        std::vector<Pos64> h64(N);
        for (int k = 0; k < N; ++k) {
            const float *v = voxel_xyz + 3 * (size_t)index(k);
            h64[k] = Pos64{v[0] * s, v[1] * s, v[2] * s, 0.0};
        }
        {
            DeviceGuard dg(p->device);
            e = plan_upload(p, &p->d_vox64, h64.data(), sizeof(Pos64) * (size_t)N);
        }
        if (e != cudaSuccess) {
            das_plan_destroy(p);
            *plan = nullptr;
            cudaGetLastError();
            return cuda_fail(e, "voxel list upload");
        }
        p->geom64.vox = p->d_vox64;
    }
    return DAS_OK;
}

das_status das_plan_set_option(das_plan p, int option, double value)
{
    if (!p) return fail(DAS_ERR_INVALID_ARG, "plan is NULL");
    switch (option) {
    case DAS_OPT_KERNEL: {
        const int k = (int)value;
        if ((double)k != value || k < DAS_KERNEL_AUTO || k > DAS_KERNEL_PAIR)
            return fail(DAS_ERR_INVALID_ARG, "invalid kernel %g", value);
        p->kernel = k;
        return DAS_OK;
    }
    case DAS_OPT_DEMOD_HZ:
        if (!std::isfinite(value)) return fail(DAS_ERR_INVALID_ARG, "f_demod must be finite");
        if (!p->is_complex() && value != 0.0)
            return fail(DAS_ERR_UNSUPPORTED, "demodulation needs a complex (IQ) plan");
        p->f_demod = value;
        p->geom.fd_over_fs = (float)(value / (double)p->fs);
        p->geom64.fd_over_fs = value / (double)p->fs;
        p->geom.rotate = value != 0.0;
        return DAS_OK;
    case DAS_OPT_TIMING:
        if (value != 0.0 && value != 1.0) return fail(DAS_ERR_INVALID_ARG, "timing must be 0 or 1");
        if (value == 1.0 && !p->ev[0]) {
            DeviceGuard dg(p->device);
            for (auto &ev : p->ev) {
                cudaError_t e = cudaEventCreate(&ev);
                if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
            }
        }
        p->timing = (int)value;
        p->timed_once = false;
        return DAS_OK;
    case DAS_OPT_STORAGE: {
        const int v = (int)value;
        if ((double)v != value || (v != DAS_STORAGE_NATIVE && v != DAS_STORAGE_F16))
            return fail(DAS_ERR_INVALID_ARG, "storage must be DAS_STORAGE_NATIVE or DAS_STORAGE_F16");
        if (v != p->storage) p->perm_zero_layout = -1;   // pad rows move with the element size
        p->storage = v;
        return DAS_OK;
    }
    case DAS_OPT_RX_GROUPS: {
        const int n = (int)value;
        if ((double)n != value || n < 0 || n > 64)
            return fail(DAS_ERR_INVALID_ARG, "receiver groups must be an integer in [0, 64]");
        p->rx_groups = n;
        return DAS_OK;
    }
    case DAS_OPT_TX_GROUPS: {
        const int n = (int)value;
        if ((double)n != value || n < 0 || n > 64)
            return fail(DAS_ERR_INVALID_ARG, "transmit groups must be an integer in [0, 64]");
        p->tx_groups = n;
        return DAS_OK;
    }
    case DAS_OPT_HOST_GROUPS: {
        const int n = (int)value;
        if ((double)n != value || n < 0 || n > 64)
            return fail(DAS_ERR_INVALID_ARG, "host groups must be an integer in [0, 64]");
        p->host_groups = n;
        return DAS_OK;
    }
    case DAS_OPT_BI_GROUP: {
        const int gsz = (int)value;
        if ((double)gsz != value || !(gsz == 0 || gsz == 2 || gsz == 4 || gsz == 8 || gsz == 16 || gsz == 32))
            return fail(DAS_ERR_INVALID_ARG, "BI group must be 0, 2, 4, 8, 16 or 32");
        p->bi_group = gsz;
        return DAS_OK;
    }
    default: return fail(DAS_ERR_INVALID_ARG, "unknown option %d", option);
    }
}

das_status das_plan_get_option(das_plan p, int option, double *value)
{
    if (!p || !value) return fail(DAS_ERR_INVALID_ARG, "NULL argument");
    switch (option) {
    case DAS_OPT_KERNEL: *value = p->kernel; return DAS_OK;
    case DAS_OPT_DEMOD_HZ: *value = p->f_demod; return DAS_OK;
    case DAS_OPT_TIMING: *value = p->timing; return DAS_OK;
    case DAS_OPT_BI_GROUP: *value = p->bi_group; return DAS_OK;
    case DAS_OPT_HOST_GROUPS: *value = p->host_groups; return DAS_OK;
    case DAS_OPT_RX_GROUPS: *value = p->rx_groups; return DAS_OK;
    case DAS_OPT_TX_GROUPS: *value = p->tx_groups; return DAS_OK;
    case DAS_OPT_STORAGE: *value = p->storage; return DAS_OK;
    default: return fail(DAS_ERR_INVALID_ARG, "unknown option %d", option);
    }
}

das_status das_plan_kernel(das_plan p, int *kernel)
{
    if (!p || !kernel) return fail(DAS_ERR_INVALID_ARG, "NULL argument");
    *kernel = resolve_kernel(p);
    return DAS_OK;
}

das_status das_plan_launches(das_plan p, int *launches)
{
    if (!p || !launches) return fail(DAS_ERR_INVALID_ARG, "NULL argument");
    const int kernel = resolve_kernel(p);
    int n = kernel == DAS_KERNEL_BL ? 0 : 1;        // the permute
    if (kernel == DAS_KERNEL_BRICK) {
        DeviceGuard dg(p->device);
        int R, T;
        brick_groups(p, R, T);
        n += R * T;
    } else {
        n += 1;
    }
    *launches = n;
    return DAS_OK;
}

das_status das_beamform(das_plan p, const void *rf, const float *tau_tx, const float *w_tx,
                        void *out, cudaStream_t stream)
{
    if (!p) return fail(DAS_ERR_INVALID_ARG, "plan is NULL");
    if (!rf || !tau_tx || !w_tx || !out) return fail(DAS_ERR_INVALID_ARG, "NULL buffer");
    if (!aligned16(rf) || !aligned16(out))
        return fail(DAS_ERR_INVALID_ARG, "rf and out must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(tau_tx) & 3u) || (reinterpret_cast<uintptr_t>(w_tx) & 3u))
        return fail(DAS_ERR_INVALID_ARG, "tau_tx and w_tx must be 4-byte aligned");
    const int kernel = resolve_kernel(p);
    das_status st = check_supported(p, kernel);
    if (st != DAS_OK) return st;
    DeviceGuard dg(p->device);
    DoneMark mark{p, stream};
    const bool cplx = p->is_complex();

    const void *src = rf;
    const bool permute = kernel != DAS_KERNEL_BL;
    const int layout = kernel == DAS_KERNEL_BI ? 3 : 2;
    if (permute) {
        das_status st2 = ensure_scratch(p, layout, stream);
        if (st2 != DAS_OK) return st2;
    }
    cudaError_t e = cudaSuccess;
    if (p->timing) e = cudaEventRecord(p->ev[0], stream);
    const bool half = p->half_rows();      // the kernels read half-precision rows
    // the pair kernel needs to know whether the record holds a non-finite sample
    unsigned *flag = kernel == DAS_KERNEL_PAIR ? p->d_flag : nullptr;
    if (e == cudaSuccess && flag) e = cudaMemsetAsync(flag, 0, sizeof(unsigned), stream);
    if (e == cudaSuccess && permute) {
        // float input with half storage is rounded on the way; half input is copied
        e = das::launch_permute(rf, p->d_perm, (int)p->elem_bytes(), p->B, p->Q, p->M, p->K,
                                layout, p->num_sms, stream, 0, -1, p->convert_half(), flag);
        src = p->d_perm;
    }
    if (e == cudaSuccess && p->timing) e = cudaEventRecord(p->ev[1], stream);
    if (e != cudaSuccess) return cuda_fail(e, "permute launch");
    switch (kernel) {
    case DAS_KERNEL_BL:
        e = p->is_double() ? das::launch_bl64(p->geom64, p->d_rx64, src, tau_tx, w_tx, out, cplx, stream)
                           : das::launch_bl(p->geom, p->d_rx, src, tau_tx, w_tx, out, cplx, stream);
        break;
    case DAS_KERNEL_BI:
        e = das::launch_bi(p->geom, p->d_rx, src, tau_tx, w_tx, out, cplx, p->bi_group, stream, half);
        break;
    case DAS_KERNEL_WINDOW:
        e = das::launch_window(p->geom, p->d_rx, src, tau_tx, w_tx, out, stream);
        break;
    case DAS_KERNEL_PAIR:
        e = das::launch_pair(p->geom, p->d_rx, src, tau_tx, w_tx, out, flag, stream);
        break;
    default: {
        // receivers in R launches of contiguous 32-receiver blocks and transmits
        // in T launches of contiguous ranges, each launch adding to y: the
        // launches' CTAs then read 1/(R T) of the record at a time
        const int blocks = (p->M + 31) / 32;
        int R, T;
        brick_groups(p, R, T);
        for (int r = 0; r < R && e == cudaSuccess; ++r) {
            const int m0 = 32 * (r * blocks / R);
            const int m1 = std::min(p->M, 32 * ((r + 1) * blocks / R));
            for (int t = 0; t < T && e == cudaSuccess; ++t)
                e = das::launch_brick(p->geom, p->d_rx, src, tau_tx, w_tx, out, cplx, stream,
                                      t * p->Q / T, (t + 1) * p->Q / T, r > 0 || t > 0, half, m0, m1);
        }
        break;
    }
    }
    if (e != cudaSuccess) return cuda_fail(e, "DAS kernel launch");
    if (p->timing) {
        e = cudaEventRecord(p->ev[2], stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
        p->timed_once = true;
        p->last_had_permute = permute;
    }
    return DAS_OK;
}

das_status das_beamform_host(das_plan p, const void *rf_host, const float *tau_tx_host,
                             const float *w_tx_host, void *out_host, cudaStream_t stream)
{
    if (!p) return fail(DAS_ERR_INVALID_ARG, "plan is NULL");
    if (!rf_host || !tau_tx_host || !w_tx_host || !out_host) return fail(DAS_ERR_INVALID_ARG, "NULL buffer");
    const int kernel = resolve_kernel(p);
    das_status st = check_supported(p, kernel);
    if (st != DAS_OK) return st;
    DeviceGuard dg(p->device);
    cudaError_t e = cudaSuccess;
    if (!p->d_rf) e = plan_alloc(p, &p->d_rf, p->rf_bytes());
    if (e == cudaSuccess && !p->d_out) e = plan_alloc(p, &p->d_out, p->out_bytes());
    if (e == cudaSuccess && !p->d_tau) e = plan_alloc(p, &p->d_tau, p->txw_bytes());
    if (e == cudaSuccess && !p->d_w) e = plan_alloc(p, &p->d_w, p->txw_bytes());
    if (e != cudaSuccess) return cuda_fail(e, "host-path device buffers");
    DoneMark mark{p, stream};
    int groups = p->host_groups > 0 ? p->host_groups : (p->Q < 5 ? p->Q : 5);
    if (kernel != DAS_KERNEL_BRICK && kernel != DAS_KERNEL_WINDOW && kernel != DAS_KERNEL_PAIR)
        groups = 1;                                  // only these kernels sum transmit ranges
    if (groups > p->Q) groups = p->Q;

    if (groups <= 1) {
        e = cudaMemcpyAsync(p->d_rf, rf_host, p->rf_bytes(), cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaMemcpyAsync(p->d_tau, tau_tx_host, p->txw_bytes(), cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaMemcpyAsync(p->d_w, w_tx_host, p->txw_bytes(), cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
        st = das_beamform(p, p->d_rf, p->d_tau, p->d_w, p->d_out, stream);
        if (st != DAS_OK) return st;
    } else {
        // Streamed: the record arrives in groups of transmits on a copy stream
        // while `stream` permutes and sums the groups already on the device.
        if (!p->copy_stream) {
            e = cudaStreamCreateWithFlags(&p->copy_stream, cudaStreamNonBlocking);
            if (e != cudaSuccess) { p->copy_stream = nullptr; return cuda_fail(e, "copy stream"); }
        }
        while ((int)p->copy_ev.size() < groups + 2) {
            cudaEvent_t ev;
            e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
            if (e != cudaSuccess) return cuda_fail(e, "copy events");
            p->copy_ev.push_back(ev);
        }
        const bool cplx = p->cplx32();
        const size_t eb = p->elem_bytes();
        const size_t plane = (size_t)p->M * p->K * eb;            // one transmit of one frame
        const size_t pitch = (size_t)p->Q * plane;                // one frame
        // nothing queued earlier on `stream` may still read the staging buffers
        e = cudaEventRecord(p->copy_ev[0], stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(p->copy_stream, p->copy_ev[0], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(p->d_tau, tau_tx_host, p->txw_bytes(), cudaMemcpyHostToDevice, p->copy_stream);
        if (e == cudaSuccess) e = cudaMemcpyAsync(p->d_w, w_tx_host, p->txw_bytes(), cudaMemcpyHostToDevice, p->copy_stream);
        if (e == cudaSuccess) e = cudaEventRecord(p->copy_ev[1], p->copy_stream);
        for (int gi = 0; gi < groups && e == cudaSuccess; ++gi) {
            const int q0 = gi * p->Q / groups, q1 = (gi + 1) * p->Q / groups;
            e = cudaMemcpy2DAsync(static_cast<char *>(p->d_rf) + q0 * plane, pitch,
                                  static_cast<const char *>(rf_host) + q0 * plane, pitch,
                                  (q1 - q0) * plane, p->B, cudaMemcpyHostToDevice, p->copy_stream);
            if (e == cudaSuccess) e = cudaEventRecord(p->copy_ev[2 + gi], p->copy_stream);
        }
        if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
        st = ensure_scratch(p, 2, stream);
        if (st != DAS_OK) return st;
        unsigned *flag = kernel == DAS_KERNEL_PAIR ? p->d_flag : nullptr;
        e = cudaStreamWaitEvent(stream, p->copy_ev[1], 0);
        if (e == cudaSuccess && flag) e = cudaMemsetAsync(flag, 0, sizeof(unsigned), stream);
        for (int gi = 0; gi < groups && e == cudaSuccess; ++gi) {
            const int q0 = gi * p->Q / groups, q1 = (gi + 1) * p->Q / groups;
            e = cudaStreamWaitEvent(stream, p->copy_ev[2 + gi], 0);
            const bool half = p->half_rows();
            if (e == cudaSuccess)
                e = das::launch_permute(p->d_rf, p->d_perm, (int)eb, p->B, p->Q, p->M, p->K, 2,
                                        p->num_sms, stream, q0, q1, p->convert_half(), flag);
            if (e == cudaSuccess)
                e = kernel == DAS_KERNEL_WINDOW
                        ? das::launch_window(p->geom, p->d_rx, p->d_perm, p->d_tau, p->d_w, p->d_out,
                                             stream, q0, q1, gi > 0)
                    : kernel == DAS_KERNEL_PAIR
                        ? das::launch_pair(p->geom, p->d_rx, p->d_perm, p->d_tau, p->d_w, p->d_out,
                                           flag, stream, q0, q1, gi > 0)
                        : das::launch_brick(p->geom, p->d_rx, p->d_perm, p->d_tau, p->d_w, p->d_out,
                                            cplx, stream, q0, q1, gi > 0, half);
        }
        if (e != cudaSuccess) return cuda_fail(e, "streamed beamform launch");
    }
    e = cudaMemcpyAsync(out_host, p->d_out, p->out_bytes(), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy");
    return DAS_OK;
}

das_status das_beamform_host_volumes(das_plan p, int n_volumes, const void *rf_host,
                                     const float *tau_tx_host, const float *w_tx_host, void *out_host,
                                     cudaStream_t stream)
{
    if (!p) return fail(DAS_ERR_INVALID_ARG, "plan is NULL");
    if (n_volumes < 1) return fail(DAS_ERR_INVALID_ARG, "n_volumes must be >= 1");
    if (!rf_host || !tau_tx_host || !w_tx_host || !out_host) return fail(DAS_ERR_INVALID_ARG, "NULL buffer");
    const int kernel = resolve_kernel(p);
    das_status st = check_supported(p, kernel);
    if (st != DAS_OK) return st;
    DeviceGuard dg(p->device);
    cudaError_t e = cudaSuccess;
    if (!p->d_rf) e = plan_alloc(p, &p->d_rf, p->rf_bytes());
    if (e == cudaSuccess && !p->d_out) e = plan_alloc(p, &p->d_out, p->out_bytes());
    if (e == cudaSuccess && !p->d_tau) e = plan_alloc(p, &p->d_tau, p->txw_bytes());
    if (e == cudaSuccess && !p->d_w) e = plan_alloc(p, &p->d_w, p->txw_bytes());
    if (e != cudaSuccess) return cuda_fail(e, "host-path device buffers");
    DoneMark mark{p, stream};
    // transmit groups as das_beamform_host streams them; kernels that cannot sum
    // transmit ranges take the record whole
    const bool ranges = kernel == DAS_KERNEL_BRICK || kernel == DAS_KERNEL_WINDOW || kernel == DAS_KERNEL_PAIR;
    int groups = !ranges ? 1 : (p->host_groups > 0 ? p->host_groups : (p->Q < 5 ? p->Q : 5));
    if (groups > p->Q) groups = p->Q;
    if (!p->copy_stream) {
        e = cudaStreamCreateWithFlags(&p->copy_stream, cudaStreamNonBlocking);
        if (e != cudaSuccess) { p->copy_stream = nullptr; return cuda_fail(e, "copy stream"); }
    }
    while ((int)p->copy_ev.size() < groups + 2) {
        cudaEvent_t ev;
        e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e, "copy events");
        p->copy_ev.push_back(ev);
    }
    while ((int)p->used_ev.size() < groups) {
        cudaEvent_t ev;
        e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e, "copy events");
        p->used_ev.push_back(ev);
    }
    const bool cplx = p->cplx32();
    const bool half = p->half_rows();
    const size_t eb = p->elem_bytes();
    const size_t plane = (size_t)p->M * p->K * eb;            // one transmit of one frame
    const size_t pitch = (size_t)p->Q * plane;                // one frame
    // nothing queued earlier on `stream` may still read the staging buffers
    e = cudaEventRecord(p->copy_ev[0], stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->copy_stream, p->copy_ev[0], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(p->d_tau, tau_tx_host, p->txw_bytes(), cudaMemcpyHostToDevice, p->copy_stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(p->d_w, w_tx_host, p->txw_bytes(), cudaMemcpyHostToDevice, p->copy_stream);
    if (e == cudaSuccess) e = cudaEventRecord(p->copy_ev[1], p->copy_stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, p->copy_ev[1], 0);
    if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
    if (ranges) {
        st = ensure_scratch(p, 2, stream);
        if (st != DAS_OK) return st;
    }
    unsigned *flag = kernel == DAS_KERNEL_PAIR ? p->d_flag : nullptr;
    for (int v = 0; v < n_volumes; ++v) {
        const char *rf_v = static_cast<const char *>(rf_host) + (size_t)v * p->rf_bytes();
        // volume v's copy of group g waits until the kernels of volume v - 1 have
        // read the staging copy of group g, then runs beside their later groups
        for (int gi = 0; gi < groups && e == cudaSuccess; ++gi) {
            const int q0 = gi * p->Q / groups, q1 = (gi + 1) * p->Q / groups;
            if (v > 0) e = cudaStreamWaitEvent(p->copy_stream, p->used_ev[gi], 0);
            if (e == cudaSuccess)
                e = cudaMemcpy2DAsync(static_cast<char *>(p->d_rf) + q0 * plane, pitch, rf_v + q0 * plane, pitch,
                                      (q1 - q0) * plane, p->B, cudaMemcpyHostToDevice, p->copy_stream);
            if (e == cudaSuccess) e = cudaEventRecord(p->copy_ev[2 + gi], p->copy_stream);
        }
        if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
        if (ranges) {
            if (flag) e = cudaMemsetAsync(flag, 0, sizeof(unsigned), stream);
            for (int gi = 0; gi < groups && e == cudaSuccess; ++gi) {
                const int q0 = gi * p->Q / groups, q1 = (gi + 1) * p->Q / groups;
                e = cudaStreamWaitEvent(stream, p->copy_ev[2 + gi], 0);
                if (e == cudaSuccess)
                    e = das::launch_permute(p->d_rf, p->d_perm, (int)eb, p->B, p->Q, p->M, p->K, 2,
                                            p->num_sms, stream, q0, q1, p->convert_half(), flag);
                if (e == cudaSuccess) e = cudaEventRecord(p->used_ev[gi], stream);
                if (e == cudaSuccess)
                    e = kernel == DAS_KERNEL_WINDOW
                            ? das::launch_window(p->geom, p->d_rx, p->d_perm, p->d_tau, p->d_w, p->d_out,
                                                 stream, q0, q1, gi > 0)
                        : kernel == DAS_KERNEL_PAIR
                            ? das::launch_pair(p->geom, p->d_rx, p->d_perm, p->d_tau, p->d_w, p->d_out,
                                               flag, stream, q0, q1, gi > 0)
                            : das::launch_brick(p->geom, p->d_rx, p->d_perm, p->d_tau, p->d_w, p->d_out,
                                                cplx, stream, q0, q1, gi > 0, half);
            }
            if (e != cudaSuccess) return cuda_fail(e, "streamed beamform launch");
        } else {
            e = cudaStreamWaitEvent(stream, p->copy_ev[2], 0);
            if (e != cudaSuccess) return cuda_fail(e, "stream wait");
            st = das_beamform(p, p->d_rf, p->d_tau, p->d_w, p->d_out, stream);
            if (st != DAS_OK) return st;
            e = cudaEventRecord(p->used_ev[0], stream);
        }
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<char *>(out_host) + (size_t)v * p->out_bytes(), p->d_out,
                                p->out_bytes(), cudaMemcpyDeviceToHost, stream);
        if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy");
    }
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "synchronise");
    return DAS_OK;
}

das_status das_plan_last_times(das_plan p, float *permute_ms, float *das_ms)
{
    if (!p || !permute_ms || !das_ms) return fail(DAS_ERR_INVALID_ARG, "NULL argument");
    if (!p->timing || !p->timed_once) return fail(DAS_ERR_INVALID_ARG, "no timed call recorded");
    DeviceGuard dg(p->device);
    cudaError_t e = cudaEventSynchronize(p->ev[2]);
    if (e == cudaSuccess) e = cudaEventElapsedTime(permute_ms, p->ev[0], p->ev[1]);
    if (e == cudaSuccess) e = cudaEventElapsedTime(das_ms, p->ev[1], p->ev[2]);
    if (e != cudaSuccess) return cuda_fail(e, "event timing");
    if (!p->last_had_permute) *permute_ms = 0.f;
    return DAS_OK;
}

das_status das_plan_device_bytes(das_plan p, size_t *bytes)
{
    if (!p || !bytes) return fail(DAS_ERR_INVALID_ARG, "NULL argument");
    size_t b = sizeof(RxPos) * p->M + p->perm_bytes + (p->d_vox ? sizeof(float4) * (size_t)p->N : 0);
    if (p->d_flag) b += 256;
    if (p->d_order) b += sizeof(int) * (size_t)p->N;
    if (p->d_rx64) b += sizeof(Pos64) * p->M;
    if (p->d_vox64) b += sizeof(Pos64) * (size_t)p->N;
    if (p->d_rf) b += p->rf_bytes();
    if (p->d_out) b += p->out_bytes();
    if (p->d_tau) b += p->txw_bytes();
    if (p->d_w) b += p->txw_bytes();
    *bytes = b;
    return DAS_OK;
}

das_status das_plan_destroy(das_plan p)
{
    if (!p) return DAS_OK;
    {
        DeviceGuard dg(p->device);
        release(p);
    }
    delete p;
    return DAS_OK;
}

das_status das_permute(const void *in, void *out, das_dtype dtype, int B, int Q, int M, int K,
                       int layout, das_storage storage, cudaStream_t stream)
{
    if (!in || !out) return fail(DAS_ERR_INVALID_ARG, "NULL buffer");
    if (dtype != DAS_F32 && dtype != DAS_C64 && dtype != DAS_F16 && dtype != DAS_C32H)
        return fail(DAS_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (B < 1 || Q < 1 || M < 1 || K < 1) return fail(DAS_ERR_INVALID_ARG, "B, Q, M, K must be >= 1");
    if ((long long)Q * M >= (1LL << 31)) return fail(DAS_ERR_INVALID_ARG, "Q*M must be < 2^31");
    if (layout < 0 || layout > 3) return fail(DAS_ERR_INVALID_ARG, "layout must be 0, 1, 2 or 3");
    if (storage != DAS_STORAGE_NATIVE && storage != DAS_STORAGE_F16)
        return fail(DAS_ERR_INVALID_ARG, "unknown storage %d", (int)storage);
    const bool half_in = dtype == DAS_F16 || dtype == DAS_C32H;
    const bool half = storage == DAS_STORAGE_F16 && !half_in;      // round float samples to half
    const size_t eb = dtype == DAS_C64 ? 8 : (dtype == DAS_F16 ? 2 : 4);
    const size_t bytes = (size_t)B * Q * M * K * eb;
    const size_t oeb = half ? eb / 2 : eb;
    if ((reinterpret_cast<uintptr_t>(in) % eb) != 0 || (reinterpret_cast<uintptr_t>(out) % oeb) != 0)
        return fail(DAS_ERR_INVALID_ARG, "in and out must be aligned to their element sizes (%zu, %zu bytes)",
                    eb, oeb);
    const size_t obytes = (size_t)B * Q * M * (K + (layout == 2 ? 3 : layout == 3 ? 2 : 0)) * oeb;
    const char *a = static_cast<const char *>(in);
    const char *b = static_cast<const char *>(out);
    if (a < b + obytes && b < a + bytes) return fail(DAS_ERR_INVALID_ARG, "in and out overlap");
    int dev = 0, sms = 1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = das::launch_permute(in, out, (int)eb, B, Q, M, K, layout, sms, stream, 0, -1, half);
    if (e != cudaSuccess) return cuda_fail(e, "permute");
    return DAS_OK;
}

das_status das_permute_bqmk_to_kqmb(const void *in, void *out, das_dtype dtype, int B, int Q, int M,
                                    int K, cudaStream_t stream)
{
    if (dtype != DAS_F32 && dtype != DAS_C64) return fail(DAS_ERR_INVALID_ARG, "dtype must be DAS_F32 or DAS_C64");
    return das_permute(in, out, dtype, B, Q, M, K, 0, DAS_STORAGE_NATIVE, stream);
}

}  // extern "C"
