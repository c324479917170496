// Lightning Indexer + top-k for callers that cannot allocate device memory.
//
// lightning_index() with scores == NULL keeps the fp32 score matrix in a
// caller-provided workspace.  Some callers have no way to provide one: a host
// program whose device memory is entirely owned by another runtime's pool
// (where a cudaMalloc of its own would fail or break that pool's accounting),
// or a latency-critical loop that must not call cudaMalloc/cudaFree because
// they can synchronise the device.  This variant keeps the score matrix in a
// fixed array compiled into the library instead.
//
// The array is a file-scope __device__ variable, so in host code its name is
// only a host-side stand-in: the device address is fetched once per device
// with cudaGetSymbolAddress (with that device current) and passed to the
// kernels as a plain pointer.
#include <mutex>

#include "lc_common.cuh"

namespace lc {

lc_status index_launch(const void *qI, const float *w, const void *kI, const lc_batch &b, int HI,
                       int dI, int m, lc_dtype dt, float *scores, int64_t ld, int32_t *dev_err,
                       cudaStream_t st);
lc_status topk_launch(const float *scores, int64_t ld, const lc_batch &b, int m, int k,
                      int32_t *topk, int32_t *dev_err, cudaStream_t st);
lc_status finish(lc_status s, cudaStream_t st, int32_t *dev_err);
bool batch_ok(const lc_batch *b);

namespace {

constexpr size_t kScratchFloats = (size_t)LC_NOALLOC_SCRATCH_BYTES / sizeof(float);

// Every call on a device shares this one array.  Each call writes every score
// it later reads (visible entries get their score, the rest of each row -inf),
// so nothing needs clearing between calls; calls that overlap on the GPU race.
__device__ __align__(256) float g_scores[kScratchFloats];

constexpr int kMaxDevices = 64;
float *g_dev_ptr[kMaxDevices];
std::mutex g_mu;

// Device address of g_scores on the current device (looked up on the first
// call on each device, with that device current, and kept for the life of the
// process: a cudaDeviceReset of that device would leave it stale).
lc_status scratch_on_current_device(float **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return LC_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return LC_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_dev_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scores);
        if (e != cudaSuccess || !p) return LC_ERR_CUDA;
        g_dev_ptr[dev] = static_cast<float *>(p);
    }
    *out = g_dev_ptr[dev];
    return LC_OK;
}

}  // namespace
}  // namespace lc

extern "C" lc_status lightning_index_topk_noalloc(const void *qI, const float *w, const void *kI,
                                                  const lc_batch *batch, int32_t HI, int32_t dI,
                                                  int32_t m, lc_dtype dtype, int32_t k,
                                                  int32_t *topk, int32_t *dev_err,
                                                  lc_stream stream) {
    using namespace lc;
    cudaStream_t st = (cudaStream_t)stream;
    if (!qI || !w || !kI || !topk || !batch_ok(batch) || m < 1 || k < 1 ||
        (dtype != LC_F32 && dtype != LC_BF16) || (reinterpret_cast<uintptr_t>(kI) & 15u) != 0)
        return LC_ERR_INVALID_ARG;
    if ((HI != 1 && HI != 2 && HI != 4 && HI != 8) || (dI != 32 && dI != 64) || k > 4096)
        return LC_ERR_UNSUPPORTED;
    // the score matrix [total_q, max_c] must fit the fixed array
    if ((double)batch->total_q * (double)batch->max_c > (double)kScratchFloats)
        return LC_ERR_WORKSPACE;
    if (batch->total_q == 0) return LC_OK;
    float *scores = nullptr;
    lc_status s = scratch_on_current_device(&scores);
    if (s != LC_OK) return s;
    const int64_t ld = batch->max_c;
    if (ld > 0) s = index_launch(qI, w, kI, *batch, HI, dI, m, dtype, scores, ld, dev_err, st);
    if (s == LC_OK) s = topk_launch(scores, ld, *batch, m, k, topk, dev_err, st);
    return finish(s, st, dev_err);
}
