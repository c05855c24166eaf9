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
//   * host code cannot use the array's name as a device address, so every
//     call looks the address up with cudaGetSymbolAddress in the current
//     context (a lookup, not an allocation).  Nothing is cached: after a
//     cudaDeviceReset, or with a non-primary context current, the next call
//     finds the array where that context has it.  The first call in a
//     context may load the library's device code there, so make it before
//     any stream capture;
//   * every call shares the one array and finds the previous call's data in
//     it.  Nothing in it has to start at zero: each region the decode kernels
//     read is written earlier in the same call.  Two calls whose work
//     overlaps on the GPU (different streams, or different host threads
//     without ordering) race on the array;
//   * sizes whose workspace would not fit are rejected with
//     QSA_ERR_UNSUPPORTED before anything is launched;
//   * nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include "qsa_common.cuh"
#include "qsa_kernels.h"

namespace {
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
}

static __device__ __align__(256) uint8_t g_decode_scratch[kNoAllocScratchBytes];

namespace {
// The device address of g_decode_scratch in the current context.
qsa_status scratch_address(void **out) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr) {
        qsa::set_error_detail("cudaGetSymbolAddress of the decode scratch array failed");
        return QSA_ERR_CUDA;
    }
    *out = p;
    return QSA_OK;
}
}  // namespace

extern "C" qsa_status qsa_sparse_attn_decode_noalloc(
    const qsa_config *cfg, int batch, const qsa_bf16 *q, const qsa_bf16 *qi, const qsa_bf16 *w,
    const qsa_bf16 *k_cache, const qsa_bf16 *v_cache, const qsa_bf16 *kblk_cache, int64_t max_ctx,
    const int32_t *seq_lens, qsa_bf16 *out, float *lse, int32_t *idx_out, int32_t *dev_status,
    void *stream) {
    // Validate every argument first, exactly as the decode with a workspace
    // does: given no workspace it returns the first argument error, or
    // QSA_ERR_WORKSPACE once every other argument is valid (its workspace
    // check comes last), and launches nothing either way.
    const qsa_status arg = qsa_sparse_attn_decode(cfg, batch, q, qi, w, k_cache, v_cache, kblk_cache,
                                                  max_ctx, seq_lens, out, lse, idx_out, nullptr, 0,
                                                  dev_status, stream);
    if (arg != QSA_ERR_WORKSPACE) return arg == QSA_OK ? QSA_ERR_INVALID_ARG : arg;
    const size_t need = qsa_decode_workspace_bytes(cfg, batch, max_ctx);
    if (need > kNoAllocScratchBytes) {
        qsa::set_error_detail(
            "this batch x max_ctx needs more decode scratch than the built-in 16 MiB; "
            "use qsa_sparse_attn_decode with a caller workspace");
        return QSA_ERR_UNSUPPORTED;
    }
    void *scratch = nullptr;
    const qsa_status st = scratch_address(&scratch);
    if (st != QSA_OK) return st;
    return qsa_sparse_attn_decode(cfg, batch, q, qi, w, k_cache, v_cache, kblk_cache, max_ctx,
                                  seq_lens, out, lse, idx_out, scratch, kNoAllocScratchBytes,
                                  dev_status, stream);
}
