// Decode step for callers that cannot allocate device memory.
//
// qsa_sparse_attn_decode needs a caller-supplied workspace.  Some callers
// have no way to provide one at the moment they run a decode step: a plain
// C host embedded in a process where another runtime owns every device
// allocation (and a raw cudaMalloc would bypass that runtime's accounting or
// exceed its budget), or a serving loop that must not allocate once it is
// running, because cudaMalloc/cudaFree can synchronise the device and can
// fail under memory pressure in the middle of a request.
//
// qsa_sparse_attn_decode_noalloc runs the same decode kernels with a fixed
// scratch area that lives in this file as a statically sized device array:
//   * the array (kNoAllocScratchBytes = 16 MiB) exists on every GPU that
//     loads this library, for as long as the library stays loaded;
//   * host code cannot use the array's name as a device address, so the
//     first call on each device (with that device current) looks up the
//     array's address with cudaGetSymbolAddress and caches it; make that
//     first call before any stream capture;
//   * every call shares the one array and finds the previous call's data in
//     it.  Nothing in it has to start at zero: each region the decode kernels
//     read is written earlier in the same call.  Two calls whose work
//     overlaps on the GPU (different streams, or different host threads
//     without ordering) race on the array;
//   * sizes whose workspace would not fit are rejected with
//     QSA_ERR_UNSUPPORTED before anything is launched;
//   * nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "qsa_common.cuh"
#include "qsa_kernels.h"

namespace {
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
}

static __device__ __align__(256) uint8_t g_decode_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_scratch_mu;
void *g_scratch_addr[64] = {};  // device address of g_decode_scratch, per device

qsa_status scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        qsa::set_error_detail("cudaGetDevice failed");
        return QSA_ERR_CUDA;
    }
    if (dev < 0 || dev >= 64) {
        qsa::set_error_detail("device ordinal out of range");
        return QSA_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || p == nullptr) {
            qsa::set_error_detail("cudaGetSymbolAddress of the decode scratch array failed");
            return QSA_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return QSA_OK;
}
}  // namespace

extern "C" qsa_status qsa_sparse_attn_decode_noalloc(
    const qsa_config *cfg, int batch, const qsa_bf16 *q, const qsa_bf16 *qi, const qsa_bf16 *w,
    const qsa_bf16 *k_cache, const qsa_bf16 *v_cache, const qsa_bf16 *kblk_cache, int64_t max_ctx,
    const int32_t *seq_lens, qsa_bf16 *out, float *lse, int32_t *idx_out, int32_t *dev_status,
    void *stream) {
    const size_t need = qsa_decode_workspace_bytes(cfg, batch, max_ctx);
    if (need > kNoAllocScratchBytes) {
        qsa::set_error_detail(
            "this batch x max_ctx needs more decode scratch than the built-in 16 MiB; "
            "use qsa_sparse_attn_decode with a caller workspace");
        return QSA_ERR_UNSUPPORTED;
    }
    void *scratch = nullptr;
    if (need > 0) {
        const qsa_status st = scratch_address(&scratch);
        if (st != QSA_OK) return st;
    }
    // need == 0 means the arguments are invalid: the call below reports why
    return qsa_sparse_attn_decode(cfg, batch, q, qi, w, k_cache, v_cache, kblk_cache, max_ctx,
                                  seq_lens, out, lse, idx_out, scratch,
                                  scratch ? kNoAllocScratchBytes : 0, dev_status, stream);
}
