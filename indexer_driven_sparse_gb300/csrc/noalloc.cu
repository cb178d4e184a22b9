// qsa_sparse_decode_noalloc: the sparse decode of qsa_sparse_decode for callers
// that cannot allocate device memory. Its split partials live in a fixed
// file-scope device array instead of a caller workspace.
//
// Who needs it: a plug-in that runs inside a host application which owns the whole
// device memory pool and hands none of it out; a process whose device memory is fully
// reserved by another allocator, so cudaMalloc would fail; and latency-critical loops
// that must not take the implicit device synchronisation an allocation can cause.
//
// The array is kNoAllocScratchBytes (16 MiB) and stays resident on every GPU that
// loads the library until the process exits. The first call on a device looks up
// the array's device address with cudaGetSymbolAddress (with that device current)
// and caches it. Calls share the
// array and each call overwrites it, so calls that overlap on the GPU (different
// streams, or concurrent graphs) race; serialise them.
#include <atomic>
#include <mutex>

#include "qsa_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mu;
std::atomic<void *> g_scratch_addr[kMaxDevices];

// Device address of g_decode_scratch on device `dev`, which must be the current device
// (set-up on first use).
qsa_status scratch_address(int dev, void **out) {
    if (dev < 0 || dev >= kMaxDevices) return qsa::host_fail(QSA_ERR_UNSUPPORTED, "device ordinal >= 64", "");
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        std::lock_guard<std::mutex> lock(g_setup_mu);
        p = g_scratch_addr[dev].load(std::memory_order_relaxed);
        if (p == nullptr) {
            const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
            if (e != cudaSuccess || p == nullptr)
                return qsa::host_fail(QSA_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed",
                                      cudaGetErrorString(e));
            g_scratch_addr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return QSA_OK;
}

}  // namespace

extern "C" QSA_API qsa_status qsa_sparse_decode_noalloc(const qsa_config *cfg, const qsa_bf16 *q,
                                                        const qsa_bf16 *k_cache, const qsa_bf16 *v_cache,
                                                        int64_t n_tokens_total, const int32_t *tok_off,
                                                        const int32_t *ctx_len, int32_t B, const int32_t *blocks,
                                                        const int32_t *count, qsa_bf16 *out, float *lse,
                                                        qsa_stream stream) {
    // Every host check runs before anything is enqueued or looked up.
    qsa_status s = qsa::sparse_decode_shape_check(cfg, B, n_tokens_total);
    if (s != QSA_OK) return s;
    const size_t need = qsa_workspace_size(QSA_OP_SPARSE_DECODE, cfg, B, 0);
    if (need > kNoAllocScratchBytes)
        return qsa::host_fail(QSA_ERR_WORKSPACE_TOO_SMALL,
                              "qsa_sparse_decode_noalloc: this batch needs more scratch than the 16 MiB static array",
                              "use qsa_sparse_decode with a caller workspace or split the batch");
    if (B == 0) return QSA_OK;
    s = qsa::sparse_decode_pointer_check(q, k_cache, v_cache, tok_off, ctx_len, blocks, count, out);
    if (s != QSA_OK) return s;
    // The array's address is per device: `stream` must belong to the current device.
    int dev = -1, stream_dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return qsa::host_fail(QSA_ERR_CUDA, "cudaGetDevice failed", cudaGetErrorString(e));
    e = cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &stream_dev);
    if (e != cudaSuccess) return qsa::host_fail(QSA_ERR_CUDA, "cudaStreamGetDevice failed", cudaGetErrorString(e));
    if (stream_dev != dev)
        return qsa::host_fail(QSA_ERR_INVALID_ARGUMENT, "qsa_sparse_decode_noalloc: stream belongs to another device",
                              "make the stream's device current before the call");
    void *scratch = nullptr;
    s = scratch_address(dev, &scratch);
    if (s != QSA_OK) return s;
    // The status block is the only part that must start at zero.
    e = cudaMemsetAsync(scratch, 0, qsa::kWsHeaderBytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return qsa::host_fail(QSA_ERR_CUDA, "cudaMemsetAsync of the status block failed",
                                                cudaGetErrorString(e));
    return qsa_sparse_decode(cfg, q, k_cache, v_cache, n_tokens_total, tok_off, ctx_len, B, blocks, count, out, lse,
                             scratch, kNoAllocScratchBytes, stream);
}
