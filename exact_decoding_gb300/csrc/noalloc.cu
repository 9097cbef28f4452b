// la_gemm_bf16_noalloc: the split-K projection GEMM for callers that cannot
// allocate device memory at call time.
//
// la_gemm_bf16 needs a caller-provided workspace when it splits K across
// CTAs.  Some callers cannot provide one: a plugin running inside a host
// framework that owns every device allocation, or a latency-critical loop in
// which cudaMalloc (and the device synchronisation it may imply) is not
// allowed.  This entry point keeps the partial sums in a fixed device array
// declared in this file instead, so a call allocates nothing: no cudaMalloc,
// no cudaFree, no allocating library routine.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it (kNoAllocScratchFloats floats, 16 MiB) until the process
// exits.  All calls share it and it keeps the last call's contents; nothing
// in it needs to start at zero, because every split writes every partial it
// later reads.  Calls whose kernels overlap on the GPU (different streams,
// or different host threads on one device) race on the array and must be
// serialised by the caller.
//
// In host code the symbol names a host-side stand-in, not a device address.
// So the first call on each device looks the address up with
// cudaGetSymbolAddress, with that device current, and caches it; that first
// call should come before any stream capture.  The cache lives as long as
// the process: after a cudaDeviceReset the cached addresses are stale.
//
// A bounded wait inside the kernel that gives up sets a bit in a second
// device word of this file; la_gemm_status reads and clears it.
#include <cstring>
#include <mutex>

#include "../../include/la.h"
#include "abi_guard.h"
#include "la_kernels.h"

static __device__ __align__(256) float g_noalloc_scratch[LA_NOALLOC_SCRATCH_FLOATS];
static __device__ __align__(256) unsigned g_noalloc_err;

namespace {

constexpr long long kNoAllocScratchFloats = LA_NOALLOC_SCRATCH_FLOATS;
constexpr int kMaxDevices = 64;

struct DevicePtrs {
    float *scratch = nullptr;
    unsigned *err = nullptr;
};
DevicePtrs g_ptrs[kMaxDevices];
std::mutex g_mu;

// Device addresses of the two symbols on the current device (looked up once).
cudaError_t symbol_ptrs(DevicePtrs *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ptrs[dev].scratch) {
        void *s = nullptr, *r = nullptr;
        e = cudaGetSymbolAddress(&s, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        e = cudaGetSymbolAddress(&r, g_noalloc_err);
        if (e != cudaSuccess) return e;
        g_ptrs[dev].scratch = static_cast<float *>(s);
        g_ptrs[dev].err = static_cast<unsigned *>(r);
    }
    *out = g_ptrs[dev];
    return cudaSuccess;
}

}  // namespace

// Address of this device's error word, or nullptr while the device has made
// no call (nothing can have set it then).
cudaError_t la::noalloc_err_word(unsigned **out) {
    *out = nullptr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    *out = g_ptrs[dev].err;
    return cudaSuccess;
}

// Read this device's error word into *bits and clear it, both on stream s
// (the caller synchronises s before reading *bits).  No allocation.
cudaError_t la::noalloc_err_take(cudaStream_t s, unsigned *bits) {
    *bits = 0;
    unsigned *w = nullptr;
    cudaError_t e = noalloc_err_word(&w);
    if (e != cudaSuccess || !w) return e;
    e = cudaMemcpyAsync(bits, w, sizeof(unsigned), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(w, 0, sizeof(unsigned), s);
    return e;
}

static int gemm_noalloc_body(const void *x, const void *w, float *y, int32_t rows, int32_t out, int32_t k,
                             int32_t splits, void *stream) {
    using namespace la;
    if (!x || !w || !y || rows < 1 || rows > 256 || out < 1 || k < 8 || k % 8 || splits < 1)
        return set_last_error(LA_ERR_INVALID_ARG, "la_gemm_bf16_noalloc: bad arguments");
    const int n_kb = (k + kBlockK - 1) / kBlockK;
    if (splits > n_kb) return set_last_error(LA_ERR_INVALID_ARG, "la_gemm_bf16_noalloc: splits > k / 64");
    if (static_cast<long long>(splits) * rows * out > kNoAllocScratchFloats)
        return set_last_error(LA_ERR_CAPACITY,
                              "la_gemm_bf16_noalloc: splits * rows * out exceeds LA_NOALLOC_SCRATCH_FLOATS");
    DevicePtrs p;
    if (symbol_ptrs(&p) != cudaSuccess)
        return set_last_error(LA_ERR_CUDA, "la_gemm_bf16_noalloc: cudaGetSymbolAddress failed");
    TcGemm g;
    std::memset(&g.p, 0, sizeof(g.p));
    const int bn = (rows + 15) / 16 * 16;
    if (make_tmap_bf16(&g.p.a[0], w, k, out, static_cast<uint64_t>(k) * 2, kBlockK, kTileM) ||
        make_tmap_bf16(&g.p.b, x, k, rows, static_cast<uint64_t>(k) * 2, kBlockK, bn))
        return set_last_error(LA_ERR_INVALID_ARG, "la_gemm_bf16_noalloc: tensor map failed (16-byte alignment?)");
    g.p.nseg = 1;
    g.p.seg_tile0[0] = 0;
    g.p.seg_tile0[1] = (out + kTileM - 1) / kTileM;
    g.p.seg_out[0] = out;
    g.p.seg_col0[0] = 0;
    g.p.n_kb = n_kb;
    g.p.splits = splits;
    g.p.nrows = rows;
    g.p.bn = bn;
    g.p.ldo = out;
    g.p.stages = tc_gemm_stages_for(bn);
    g.p.split_stride = static_cast<long long>(rows) * out;
    g.p.out = splits > 1 ? p.scratch : y;
    g.p.err = p.err;
    tc_gemm_finalize(g);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (tc_gemm_launch(g, s) != cudaSuccess) return set_last_error(LA_ERR_CUDA, "la_gemm_bf16_noalloc: launch failed");
    if (splits > 1 && reduce_splits_launch(p.scratch, splits, g.p.split_stride, rows, out, y, s) != cudaSuccess)
        return set_last_error(LA_ERR_CUDA, "la_gemm_bf16_noalloc: reduce launch failed");
    return LA_OK;
}

extern "C" int la_gemm_bf16_noalloc(const void *x, const void *w, float *y, int32_t rows, int32_t out, int32_t k,
                                    int32_t splits, void *stream) {
    return la::abi_guard("la_gemm_bf16_noalloc",
                         [&] { return gemm_noalloc_body(x, w, y, rows, out, k, splits, stream); });
}
