// The extern "C" boundary of libqsa.so: argument validation, workspace
// carving, TMA tensor maps, and the launch sequence of each entry point.
// Declarations and their documentation are in include/qsa.h.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "qsa_common.cuh"
#include "qsa_kernels.h"

namespace {

thread_local std::string g_detail = "no error";

qsa_status fail(qsa_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
qsa_status fail(qsa_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_detail = buf;
    return s;
}

qsa_status cuda_fail(cudaError_t e, const char *where) {
    return fail(QSA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

qsa_status ok() {
    g_detail = "no error";
    return QSA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// per-device SM count, cached
int sm_count() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D bf16 tensor [rows, inner] row-major, 128-byte swizzled boxes of
// [box_rows, 64] (out-of-range rows read as zero).
qsa_status make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows,
                    uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return fail(QSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(QSA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return QSA_OK;
}

// 5-D bf16 map of K' or V laid out [nseq][rows][2 heads][256 dims]: dims
// {64 dims, rows, 2 heads, 4 dim chunks, nseq} (strides 1024, 512, 128,
// rows * 1024 bytes), box {64, 4, 2, 4, 1} = one 4-token block of both heads,
// dim chunk outermost, 128-byte swizzle; rows past the end read as zeros.
qsa_status make_kv_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t nseq) {
    auto fn = encode_fn();
    if (!fn) return fail(QSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[5] = {64, rows, 2, 4, nseq};
    cuuint64_t strides[4] = {1024, 512, 128, rows * 1024};
    cuuint32_t box[5] = {64, 4, 2, 4, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(QSA_ERR_CUDA, "cuTensorMapEncodeTiled (K/V) failed (%d)", static_cast<int>(r));
    return QSA_OK;
}

// Which attention kernel runs: the warp-MMA kernel (default: the faster of
// the two as measured) or, with the environment variable
// QSA_ATTENTION_KERNEL=tc set when the library is first used, the tcgen05
// kernel (sparse_attn_tc.cu).  Both compute the same attention.
bool use_tc_attention() {
    static const bool tc = [] {
        const char *v = std::getenv("QSA_ATTENTION_KERNEL");
        return v && std::strcmp(v, "tc") == 0;
    }();
    return tc;
}

// Prefill attention of a.L query rows at positions a.q_off.., keys from the
// first key_rows rows of a.k / a.v.
qsa_status attention_prefill(const qsa::AttnArgs &a, const qsa::RopeFreqs &freqs, int64_t key_rows,
                             cudaStream_t s) {
    cudaError_t e;
    if (use_tc_attention()) {
        CUtensorMap mk, mv;
        qsa_status st = make_kv_map(&mk, a.k, static_cast<uint64_t>(key_rows), 1);
        if (st != QSA_OK) return st;
        st = make_kv_map(&mv, a.v, static_cast<uint64_t>(key_rows), 1);
        if (st != QSA_OK) return st;
        e = qsa::launch_attn_prefill_tc(a, freqs, mk, mv, key_rows, s);
    } else {
        e = qsa::launch_attn_prefill(a, freqs, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    return QSA_OK;
}

qsa_status check_cfg(const qsa_config *cfg) {
    if (!cfg) return fail(QSA_ERR_INVALID_ARG, "cfg is NULL");
    if (cfg->block_size != qsa::kBlock || cfg->n_q_heads != qsa::kHQ ||
        cfg->n_kv_heads != qsa::kHKV || cfg->head_dim != qsa::kD || cfg->rope_dim != qsa::kRD ||
        cfg->n_idx_heads != qsa::kHI || cfg->idx_dim != qsa::kDI)
        return fail(QSA_ERR_UNSUPPORTED,
                    "only block 4, 24/2 heads of dim 256, rope dim 64, indexer 4 x 128 are compiled in");
    if (cfg->budget_blocks < 1) return fail(QSA_ERR_INVALID_ARG, "budget_blocks must be >= 1");
    if (cfg->budget_blocks > qsa::kMaxBudget)
        return fail(QSA_ERR_UNSUPPORTED, "budget_blocks > %d", qsa::kMaxBudget);
    if (!(cfg->rope_theta > 0.0) || !std::isfinite(cfg->rope_theta))
        return fail(QSA_ERR_INVALID_ARG, "rope_theta must be finite and > 0");
    if (!std::isfinite(cfg->softmax_scale))
        return fail(QSA_ERR_INVALID_ARG, "softmax_scale must be finite");
    if (!std::isfinite(cfg->yarn_factor))
        return fail(QSA_ERR_INVALID_ARG, "yarn_factor must be finite");
    if (cfg->yarn_factor > 1.f &&
        (cfg->yarn_original_max_pos < 1 || !(cfg->yarn_alpha >= 0.f) || !(cfg->yarn_beta > cfg->yarn_alpha) ||
         !std::isfinite(cfg->yarn_beta)))
        return fail(QSA_ERR_INVALID_ARG, "YaRN needs original_max_pos >= 1 and 0 <= alpha < beta");
    return QSA_OK;
}

// Rotary frequencies theta^(-2i/64), rescaled by YaRN when it is on: with
// r = original context / wavelength, frequencies with r above beta keep their
// value, those below alpha are divided by the factor, and a linear ramp in r
// blends the two in between (model card "Processing Ultra-Long Texts"; the
// published YaRN method).
qsa::RopeFreqs freqs_of(const qsa_config *cfg) {
    qsa::RopeFreqs f;
    const bool yarn = cfg->yarn_factor > 1.f;
    for (int i = 0; i < 32; ++i) {
        const double w = std::pow(cfg->rope_theta, -2.0 * i / qsa::kRD);
        if (!yarn) {
            f.inv_freq[i] = w;
            continue;
        }
        const double ratio = static_cast<double>(cfg->yarn_original_max_pos) * w / (2.0 * 3.14159265358979323846);
        const double a = cfg->yarn_alpha, b = cfg->yarn_beta;
        double keep = (ratio - a) / (b - a);  // share of the original frequency
        keep = keep < 0.0 ? 0.0 : (keep > 1.0 ? 1.0 : keep);
        f.inv_freq[i] = keep * w + (1.0 - keep) * (w / cfg->yarn_factor);
    }
    return f;
}

// Softmax scale in the log2 domain; YaRN multiplies the logits by
// (0.1 ln s + 1)^2 (its temperature on both queries and keys).
float scale_log2_of(const qsa_config *cfg) {
    double sc = cfg->softmax_scale > 0.f ? cfg->softmax_scale : 1.0 / std::sqrt(double(qsa::kD));
    if (cfg->yarn_factor > 1.f) {
        const double m = 0.1 * std::log(static_cast<double>(cfg->yarn_factor)) + 1.0;
        sc *= m * m;
    }
    return static_cast<float>(sc * 1.4426950408889634);
}

#define REQ_PTR(p)                                                                       \
    do {                                                                                 \
        if (!(p)) return fail(QSA_ERR_INVALID_ARG, "%s is NULL", #p);                    \
        if (!aligned16(p)) return fail(QSA_ERR_INVALID_ARG, "%s is not 16-byte aligned", #p); \
    } while (0)
#define OPT_PTR(p)                                                                       \
    do {                                                                                 \
        if ((p) && !aligned16(p))                                                        \
            return fail(QSA_ERR_INVALID_ARG, "%s is not 16-byte aligned", #p);           \
    } while (0)

constexpr int64_t kMaxL = int64_t(1) << 24;           // tokens per prefill call
constexpr int64_t kMaxScoresL = 65536;
constexpr int64_t kMaxDecodeCtx = int64_t(47) * 16384 * 4;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t index_ws(int64_t L) {
    const size_t kblk = align_up(static_cast<size_t>(L / qsa::kBlock) * qsa::kDI * 2 + 16, 1024);
    return kblk + qsa::index_cand_bytes(L, sm_count());
}

}  // namespace

namespace qsa {
// Lets other translation units of the library set the message returned by
// qsa_last_error_detail().
void set_error_detail(const char *msg) { g_detail = msg; }
}  // namespace qsa

// ------------------------------------------------- overlapped prefill --
// The indexer is bound by its epilogue's instruction issue and the
// attention by HBM bytes, so the two can share the GPU: the query rows are
// cut into chunks, and while the attention of chunk j-1 runs on part of the
// SMs, the indexer of chunk j runs as a persistent grid on the others (a
// second, higher-priority stream).  The split balances the two stages' time
// per chunk from per-SM costs fitted to B300 runs of both kernels, side by
// side, at 128K and 1M tokens: the indexer takes 2.14e-10 SM-seconds per
// (query, past block) pair plus 8.2e-6 per query row (its list start-up and
// final selection); the attention consumes 75 GB/s of gathered K/V per SM
// (2 KiB per attended key) and cannot go faster than 8.3 TB/s of gathered
// bytes for the whole GPU (its rate alone at 1M, above the HBM copy rate
// because blocks that nearby queries share are read from L2).  Where K/V
// sits in L2 more (topic-segment inputs) the attention runs faster than
// that and the indexer's share of the SMs sets the time, so the costs lean
// towards the indexer; at 1M tokens (ms, i.i.d. / topic segments): 70 GB/s
// per SM 658-663 / 658, 75: 662-665 / 638, 80 with 9 TB/s: 668-670 / 619,
// 90 with 10 TB/s: 675 / 592, and the earlier 65 with 6.9 TB/s 665-670 /
// 697.
// Below 256K tokens the attention's K/V mostly sits in L2 and the attention
// is bound by its SMs rather than by HBM, so there is nothing to hand to the
// indexer: shorter prefills run the two stages one after the other.
namespace {

constexpr int64_t kOverlapMinL = 262144;
constexpr int kEdgeParts = 4;  // parts of the first and of the last chunk

constexpr double kIdxPairSm = 2.14e-10;
constexpr double kIdxRowSm = 8.2e-6;
constexpr double kAttnKeySm = 2048.0 / 75e9;
constexpr double kAttnKeyFloor = 2048.0 / 8.3e12;

// sum over t in [r0, r1) of floor(t/4): the pairs the indexer scores
double pairs_in(int64_t r0, int64_t r1) {
    auto upto = [](int64_t n) {  // sum over t < n of floor(t/4)
        const int64_t q = n / 4, r = n % 4;
        return 4.0 * (static_cast<double>(q) * (q - 1) / 2.0) + static_cast<double>(r) * q;
    };
    return upto(r1) - upto(r0);
}

// sum over t in [r0, r1) of the keys query t attends: t+1 while its block
// is below the budget, 4(budget-1) + t%4 + 1 after that
double keys_in(int64_t r0, int64_t r1, int budget) {
    const int64_t t0 = 4 * static_cast<int64_t>(budget - 1);
    double s = 0.0;
    const int64_t a1 = r1 < t0 ? r1 : t0;
    if (r0 < a1) s += (static_cast<double>(a1) * (a1 + 1) - static_cast<double>(r0) * (r0 + 1)) / 2.0;
    const int64_t b0 = r0 > t0 ? r0 : t0;
    if (b0 < r1) s += static_cast<double>(r1 - b0) * (4.0 * (budget - 1) + 2.5);
    return s;
}

}  // namespace

extern "C" {

void qsa_default_config(qsa_config *cfg) {
    if (!cfg) return;
    cfg->block_size = qsa::kBlock;
    cfg->budget_blocks = qsa::kMaxBudget;
    cfg->n_q_heads = qsa::kHQ;
    cfg->n_kv_heads = qsa::kHKV;
    cfg->head_dim = qsa::kD;
    cfg->rope_dim = qsa::kRD;
    cfg->n_idx_heads = qsa::kHI;
    cfg->idx_dim = qsa::kDI;
    cfg->rope_theta = 1.0e7;
    cfg->softmax_scale = 1.0f / 16.0f;
    cfg->yarn_factor = 1.0f;  // off; the model card's setting is 4
    cfg->yarn_original_max_pos = 262144;
    cfg->yarn_alpha = 1.0f;
    cfg->yarn_beta = 32.0f;
}

const char *qsa_status_string(qsa_status s) {
    switch (s) {
        case QSA_OK: return "QSA_OK";
        case QSA_ERR_INVALID_ARG: return "QSA_ERR_INVALID_ARG";
        case QSA_ERR_UNSUPPORTED: return "QSA_ERR_UNSUPPORTED";
        case QSA_ERR_WORKSPACE: return "QSA_ERR_WORKSPACE";
        case QSA_ERR_CUDA: return "QSA_ERR_CUDA";
        case QSA_ERR_TIMEOUT: return "QSA_ERR_TIMEOUT";
        case QSA_ERR_DEVICE_CHECK: return "QSA_ERR_DEVICE_CHECK";
    }
    return "QSA_ERR_UNKNOWN";
}

const char *qsa_last_error_detail(void) { return g_detail.c_str(); }

qsa_status qsa_kprep(const qsa_config *cfg, int batch, int64_t L, int64_t max_ctx,
                     const qsa_bf16 *ki, const qsa_bf16 *k, qsa_bf16 *k_rot, qsa_bf16 *kblk,
                     void *stream) {
    qsa_status st = check_cfg(cfg);
    if (st != QSA_OK) return st;
    if (batch < 1) return fail(QSA_ERR_INVALID_ARG, "batch must be >= 1");
    if (L < 1 || max_ctx < L) return fail(QSA_ERR_INVALID_ARG, "need 1 <= L <= max_ctx");
    if (max_ctx > (int64_t(1) << 40) / batch) return fail(QSA_ERR_UNSUPPORTED, "too many tokens");
    REQ_PTR(ki);
    REQ_PTR(kblk);
    if ((k == nullptr) != (k_rot == nullptr))
        return fail(QSA_ERR_INVALID_ARG, "k and k_rot must both be given or both be NULL");
    OPT_PTR(k);
    OPT_PTR(k_rot);
    if (batch > 1 && (max_ctx % qsa::kBlock) != 0 && L / qsa::kBlock > 0)
        return fail(QSA_ERR_INVALID_ARG, "max_ctx must be a multiple of 4 for batch > 1");
    cudaError_t e = qsa::launch_kprep(batch, 0, L, max_ctx, ki, k, k_rot, kblk, freqs_of(cfg), sm_count(),
                                      static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kprep launch");
    return ok();
}

size_t qsa_index_topk_workspace_bytes(const qsa_config *cfg, int64_t L) {
    if (check_cfg(cfg) != QSA_OK || L < 1 || L > kMaxL) return 0;
    return index_ws(L);
}

static qsa_status index_common(const qsa_config *cfg, const qsa_bf16 *qi, const qsa_bf16 *w,
                               const qsa_bf16 *ki, const qsa_bf16 *k, qsa_bf16 *k_rot, int64_t L,
                               int32_t *idx, float *score, float *dense, void *ws,
                               size_t ws_bytes, int32_t *dev_status, void *stream) {
    qsa_status st = check_cfg(cfg);
    if (st != QSA_OK) return st;
    if (L < 1) return fail(QSA_ERR_INVALID_ARG, "L must be >= 1");
    if (L > kMaxL) return fail(QSA_ERR_UNSUPPORTED, "L > %lld", static_cast<long long>(kMaxL));
    REQ_PTR(qi);
    REQ_PTR(w);
    REQ_PTR(ki);
    REQ_PTR(dev_status);
    if ((k == nullptr) != (k_rot == nullptr))
        return fail(QSA_ERR_INVALID_ARG, "k and k_rot must both be given or both be NULL");
    OPT_PTR(k);
    OPT_PTR(k_rot);
    if (dense) {
        REQ_PTR(dense);
    } else {
        REQ_PTR(idx);
        OPT_PTR(score);
    }
    const size_t need = index_ws(L);
    if (!ws || ws_bytes < need)
        return fail(QSA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, ws_bytes);
    if (!aligned16(ws)) return fail(QSA_ERR_INVALID_ARG, "ws is not 16-byte aligned");

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int sms = sm_count();
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    // TMA needs a 16-byte aligned base; round the block-key region up to 1 KiB
    uint16_t *kblk = reinterpret_cast<uint16_t *>(align_up(reinterpret_cast<uintptr_t>(wsb), 16));
    const size_t kblk_bytes = align_up(static_cast<size_t>(L / qsa::kBlock) * qsa::kDI * 2 + 16, 1024);
    void *cand = wsb + kblk_bytes;

    cudaError_t e = qsa::launch_kprep(1, 0, L, L, ki, k, k_rot, kblk, freqs_of(cfg), sms, s);
    if (e != cudaSuccess) return cuda_fail(e, "kprep launch");
    if (!dense && cfg->budget_blocks == 1) {
        e = qsa::launch_fill_current_only(0, L, qsa::kBlock, 1, idx, score, s);
        if (e != cudaSuccess) return cuda_fail(e, "selection launch");
        return ok();
    }
    CUtensorMap map_q, map_k;
    st = make_map(&map_q, qi, qsa::kDI, static_cast<uint64_t>(L) * qsa::kHI, 256);
    if (st != QSA_OK) return st;
    const int64_t nbk = L / qsa::kBlock;
    st = make_map(&map_k, kblk, qsa::kDI, static_cast<uint64_t>(nbk > 0 ? nbk : 1), 128);
    if (st != QSA_OK) return st;
    int *stop = qsa::index_stop_word(cand, qsa::index_cand_bytes(L, sms));
    e = cudaMemsetAsync(stop, 0, sizeof(int), s);
    if (e != cudaSuccess) return cuda_fail(e, "memset");
    e = qsa::launch_index(map_q, map_k, 0, L, qsa::kBlock, cfg->budget_blocks, w, idx, score, dense, cand,
                          dev_status, sms, stop, s);
    if (e != cudaSuccess) return cuda_fail(e, "indexer launch");
    return ok();
}

qsa_status qsa_index_topk(const qsa_config *cfg, const qsa_bf16 *qi, const qsa_bf16 *w,
                          const qsa_bf16 *ki, const qsa_bf16 *k, qsa_bf16 *k_rot, int64_t L,
                          int32_t *idx, float *score, void *ws, size_t ws_bytes,
                          int32_t *dev_status, void *stream) {
    return index_common(cfg, qi, w, ki, k, k_rot, L, idx, score, nullptr, ws, ws_bytes,
                        dev_status, stream);
}

qsa_status qsa_index_scores(const qsa_config *cfg, const qsa_bf16 *qi, const qsa_bf16 *w,
                            const qsa_bf16 *ki, int64_t L, float *scores, void *ws,
                            size_t ws_bytes, int32_t *dev_status, void *stream) {
    if (L > kMaxScoresL) return fail(QSA_ERR_UNSUPPORTED, "dense scores need L <= %lld",
                                     static_cast<long long>(kMaxScoresL));
    if (!scores) return fail(QSA_ERR_INVALID_ARG, "scores is NULL");
    return index_common(cfg, qi, w, ki, nullptr, nullptr, L, nullptr, nullptr, scores, ws, ws_bytes,
                        dev_status, stream);
}

qsa_status qsa_sparse_attn_prefill_cached(const qsa_config *cfg, const qsa_bf16 *q,
                                          const qsa_bf16 *k_rot, const qsa_bf16 *v, const int32_t *idx,
                                          int64_t q_offset, int64_t Lq, qsa_bf16 *out, float *lse,
                                          int32_t *dev_status, void *stream) {
    qsa_status st = check_cfg(cfg);
    if (st != QSA_OK) return st;
    if (Lq < 1) return fail(QSA_ERR_INVALID_ARG, "the number of query rows must be >= 1");
    if (q_offset < 0) return fail(QSA_ERR_INVALID_ARG, "q_offset must be >= 0");
    if (q_offset + Lq > kMaxL) return fail(QSA_ERR_UNSUPPORTED, "more than %lld positions", static_cast<long long>(kMaxL));
    REQ_PTR(q);
    REQ_PTR(k_rot);
    REQ_PTR(v);
    REQ_PTR(idx);
    REQ_PTR(out);
    OPT_PTR(lse);
    REQ_PTR(dev_status);
    qsa::AttnArgs a{};
    a.q = q;
    a.k = k_rot;
    a.v = v;
    a.seq_stride = 0;
    a.idx = idx;
    a.budget = cfg->budget_blocks;
    a.seq_lens = nullptr;
    a.L = Lq;
    a.q_off = q_offset;
    a.out = out;
    a.lse = lse;
    a.nsplit = 1;
    a.scale_log2 = scale_log2_of(cfg);
    a.status = dev_status;
    st = attention_prefill(a, freqs_of(cfg), q_offset + Lq, static_cast<cudaStream_t>(stream));
    if (st != QSA_OK) return st;
    return ok();
}

qsa_status qsa_sparse_attn_prefill(const qsa_config *cfg, const qsa_bf16 *q,
                                   const qsa_bf16 *k_rot, const qsa_bf16 *v, const int32_t *idx,
                                   int64_t L, qsa_bf16 *out, float *lse, int32_t *dev_status,
                                   void *stream) {
    return qsa_sparse_attn_prefill_cached(cfg, q, k_rot, v, idx, 0, L, out, lse, dev_status, stream);
}

// The indexer's SMs for a chunk whose indexer work is w SM-s, run beside an
// attention chunk of a SM-s that cannot take less than fl seconds: the x
// that minimises the later of the two to finish.
int best_split(double w, double a, double fl, int sms) {
    int best = 1;
    double best_t = 1e300;
    for (int x = 1; x < sms; ++x) {
        const double ta = a / (sms - x) > fl ? a / (sms - x) : fl;
        const double t = w / x > ta ? w / x : ta;
        if (t < best_t) {
            best_t = t;
            best = x;
        }
    }
    return best;
}
double chunk_index_work(const int64_t *b, int j) {
    return pairs_in(b[j], b[j + 1]) * kIdxPairSm + static_cast<double>(b[j + 1] - b[j]) * kIdxRowSm;
}
double chunk_attn_keys(const int64_t *b, int j, int budget) { return keys_in(b[j], b[j + 1], budget); }

int qsa_prefill_overlap_plan(const qsa_config *cfg, int64_t L, int sms, int max_chunks,
                             int64_t *chunk_begin, int *index_ctas) {
    if (check_cfg(cfg) != QSA_OK || L < 1 || L > kMaxL || sms < 2 || max_chunks < 1 || !chunk_begin ||
        !index_ctas)
        return 0;
    const int64_t tq = 64;  // query rows per indexer tile
    int64_t rows = ((L + 15) / 16 + tq - 1) / tq * tq;
    if (rows < 16384) rows = 16384;
    // equal chunks; a remainder under half a chunk joins the last one
    int64_t n = (L + rows / 2) / rows;
    if (n < 1) n = 1;
    if (n > max_chunks) {
        rows = ((L + max_chunks - 1) / max_chunks + tq - 1) / tq * tq;
        n = (L + rows - 1) / rows;
    }
    if (cfg->budget_blocks <= 1 || L < kOverlapMinL) n = 1;
    if (n <= 1) {
        chunk_begin[0] = 0;
        chunk_begin[1] = L;
        index_ctas[0] = sms;
        return 1;
    }
    // the first and the last chunk in kEdgeParts parts each (64-row tiles):
    // only the first part's indexer runs alone, and only the last part's
    // attention, so the pipeline fills and drains in a quarter of a chunk
    int64_t m = 0;
    const bool split = n >= 2 && rows / kEdgeParts >= tq && n + 2 * (kEdgeParts - 1) <= max_chunks;
    for (int64_t j = 0; j < n; ++j) {
        const int64_t a = j * rows, b = j + 1 < n ? (j + 1) * rows : L;
        const int parts = split && (j == 0 || j == n - 1) ? kEdgeParts : 1;
        const int64_t step = ((b - a) / parts) / tq * tq;
        for (int k = 0; k < parts; ++k) chunk_begin[m++] = a + k * step;
    }
    n = m;
    chunk_begin[n] = L;
    index_ctas[0] = sms;  // the first chunk's indexer runs alone
    for (int j = 1; j < static_cast<int>(n); ++j) {
        const double keys = chunk_attn_keys(chunk_begin, j - 1, cfg->budget_blocks);
        index_ctas[j] = best_split(chunk_index_work(chunk_begin, j), keys * kAttnKeySm, keys * kAttnKeyFloor, sms);
    }
    return static_cast<int>(n);
}

size_t qsa_prefill_overlapped_workspace_bytes(const qsa_config *cfg, int64_t L) {
    return qsa_index_topk_workspace_bytes(cfg, L);
}

qsa_status qsa_prefill_overlapped(const qsa_config *cfg, const qsa_bf16 *q, const qsa_bf16 *qi,
                                  const qsa_bf16 *w, const qsa_bf16 *ki, const qsa_bf16 *k, qsa_bf16 *k_rot,
                                  const qsa_bf16 *v, int64_t L, int32_t *idx, float *score, qsa_bf16 *out,
                                  float *lse, void *ws, size_t ws_bytes, int32_t *dev_status, void *stream) {
    qsa_status st = check_cfg(cfg);
    if (st != QSA_OK) return st;
    if (L < 1) return fail(QSA_ERR_INVALID_ARG, "L must be >= 1");
    if (L > kMaxL) return fail(QSA_ERR_UNSUPPORTED, "L > %lld", static_cast<long long>(kMaxL));
    REQ_PTR(q);
    REQ_PTR(qi);
    REQ_PTR(w);
    REQ_PTR(ki);
    REQ_PTR(k);
    REQ_PTR(k_rot);
    REQ_PTR(v);
    REQ_PTR(idx);
    OPT_PTR(score);
    REQ_PTR(out);
    OPT_PTR(lse);
    REQ_PTR(dev_status);
    const size_t need = index_ws(L);
    if (!ws || ws_bytes < need)
        return fail(QSA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, ws_bytes);
    if (!aligned16(ws)) return fail(QSA_ERR_INVALID_ARG, "ws is not 16-byte aligned");

    const int sms = sm_count();
    constexpr int kMaxChunks = 64;
    int64_t begin[kMaxChunks + 1];
    int ctas[kMaxChunks];
    int n = qsa_prefill_overlap_plan(cfg, L, sms, kMaxChunks, begin, ctas);
    if (n < 1) return fail(QSA_ERR_INVALID_ARG, "no chunk plan");
    // a stream being captured into a CUDA graph gets the serial schedule (no
    // helper stream is created while a capture is open)
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t ce = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cap);
    if (ce != cudaSuccess) return cuda_fail(ce, "stream capture query");
    if (cap != cudaStreamCaptureStatusNone) n = 1;
    if (n == 1) {  // nothing to overlap: the two stages one after the other
        st = index_common(cfg, qi, w, ki, k, k_rot, L, idx, score, nullptr, ws, ws_bytes, dev_status, stream);
        if (st != QSA_OK) return st;
        return qsa_sparse_attn_prefill_cached(cfg, q, k_rot, v, idx, 0, L, out, lse, dev_status, stream);
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    uint16_t *kblk = reinterpret_cast<uint16_t *>(wsb);
    const size_t kblk_bytes = align_up(static_cast<size_t>(L / qsa::kBlock) * qsa::kDI * 2 + 16, 1024);
    void *cand = wsb + kblk_bytes;
    const int budget = cfg->budget_blocks;
    const qsa::RopeFreqs freqs = freqs_of(cfg);

    // the side stream and the events live until their work is done (CUDA
    // releases a destroyed stream or event once its pending work completes)
    int lo = 0, hi = 0;
    cudaError_t e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
    if (e != cudaSuccess) return cuda_fail(e, "stream priority range");
    cudaStream_t side = nullptr;
    e = cudaStreamCreateWithPriority(&side, cudaStreamNonBlocking, hi);
    if (e != cudaSuccess) return cuda_fail(e, "side stream");
    // per chunk: the indexer's start and end on the side stream, the
    // attention's start and end on `stream`; then the K-prep's end
    cudaEvent_t ev[4 * kMaxChunks + 1];
    cudaEvent_t *ti0 = ev, *ti1 = ev + n, *ta0 = ev + 2 * n, *ta1 = ev + 3 * n, *kp = ev + 4 * n;
    int nev = 0;
    auto cleanup = [&]() {
        for (int i = 0; i < nev; ++i) cudaEventDestroy(ev[i]);
        cudaStreamDestroy(side);
    };
    for (; nev < 4 * n + 1; ++nev) {
        e = cudaEventCreate(&ev[nev]);
        if (e != cudaSuccess) {
            cleanup();
            return cuda_fail(e, "event");
        }
    }
    int *stop = qsa::index_stop_word(cand, qsa::index_cand_bytes(L, sms));
    auto enqueue_index = [&](int j) -> qsa_status {
        const int64_t r0 = begin[j], nr = begin[j + 1] - begin[j];
        CUtensorMap map_q, map_k;
        qsa_status st2 = make_map(&map_q, qi + r0 * qsa::kHI * qsa::kDI, qsa::kDI,
                                  static_cast<uint64_t>(nr) * qsa::kHI, 256);
        if (st2 != QSA_OK) return st2;
        const int64_t nbk = (r0 + nr) / qsa::kBlock;
        st2 = make_map(&map_k, kblk, qsa::kDI, static_cast<uint64_t>(nbk > 0 ? nbk : 1), 128);
        if (st2 != QSA_OK) return st2;
        cudaError_t e2 = cudaEventRecord(ti0[j], side);
        if (e2 != cudaSuccess) return cuda_fail(e2, "event record");
        e2 = qsa::launch_index(map_q, map_k, r0, nr, qsa::kBlock, budget, w + r0 * qsa::kHI, idx + r0 * budget,
                               score ? score + r0 * budget : nullptr, nullptr, cand, dev_status, ctas[j], stop,
                               side);
        if (e2 != cudaSuccess) return cuda_fail(e2, "indexer launch");
        if ((e2 = cudaEventRecord(ti1[j], side)) != cudaSuccess) return cuda_fail(e2, "event record");
        return QSA_OK;
    };
    auto enqueue_attn = [&](int j) -> qsa_status {
        const int64_t r0 = begin[j], nr = begin[j + 1] - begin[j];
        cudaError_t e2 = cudaStreamWaitEvent(s, ti1[j], 0);
        if (e2 != cudaSuccess) return cuda_fail(e2, "stream wait");
        if ((e2 = cudaEventRecord(ta0[j], s)) != cudaSuccess) return cuda_fail(e2, "event record");
        qsa::AttnArgs a{};
        a.q = q + r0 * qsa::kHQ * qsa::kD;
        a.k = k_rot;
        a.v = v;
        a.idx = idx + r0 * budget;
        a.budget = budget;
        a.L = nr;
        a.q_off = r0;
        a.out = out + r0 * qsa::kHQ * qsa::kD;
        a.lse = lse ? lse + r0 * qsa::kHQ : nullptr;
        a.nsplit = 1;
        a.scale_log2 = scale_log2_of(cfg);
        a.status = dev_status;
        qsa_status st3 = attention_prefill(a, freqs, L, s);
        if (st3 != QSA_OK) return st3;
        if ((e2 = cudaEventRecord(ta1[j], s)) != cudaSuccess) return cuda_fail(e2, "event record");
        return QSA_OK;
    };
    // The split adapts while the call runs.  Before chunk j's indexer is
    // enqueued, the host waits for the pair that ran side by side before it
    // (the indexer of chunk j-1 and the attention of chunk j-2), rescales
    // each stage's cost halfway (in the log) towards what that pair took,
    // and picks chunk j's split from the rescaled costs; then it enqueues
    // chunk j's indexer and chunk j-1's attention, in that order, so the
    // indexer (on the higher-priority stream) takes its SMs before the
    // attention's CTAs fill the GPU, and each indexer chunk starts with the
    // attention it is paired with, as the cost model assumes.  Where the
    // attention's K/V sits in L2 more than the fitted costs expect
    // (topic-segment inputs) the later chunks give the indexer more SMs.
    // Measured at 1M tokens (ms, i.i.d. / topic segments, three boxes): 660-666
    // / 599 against 663-672 / 633-634 with the fixed plan; letting the host
    // run two or three chunks ahead 664 / 597 and 668-671 / 602; enqueuing
    // the attention before the wait 673-674 / 596 (its CTAs took the SMs
    // first).
    constexpr int kLookahead = 1;
    double s_idx = 1.0, s_att = 1.0;
    auto clampd = [](double v, double lo_, double hi_) { return v < lo_ ? lo_ : (v > hi_ ? hi_ : v); };
    auto adapt = [&](int j) -> qsa_status {
        const int k2 = j - kLookahead;  // the newest pair that can have finished
        if (k2 < 2) return QSA_OK;
        cudaError_t e2 = cudaEventSynchronize(ti1[k2]);
        if (e2 == cudaSuccess) e2 = cudaEventSynchronize(ta1[k2 - 1]);
        if (e2 != cudaSuccess) return cuda_fail(e2, "event wait");
        float t_i = 0.f, t_a = 0.f;
        if (cudaEventElapsedTime(&t_i, ti0[k2], ti1[k2]) != cudaSuccess ||
            cudaEventElapsedTime(&t_a, ta0[k2 - 1], ta1[k2 - 1]) != cudaSuccess || t_i <= 0.f || t_a <= 0.f)
            return QSA_OK;  // no usable times: keep the costs
        const double keys = chunk_attn_keys(begin, k2 - 1, budget);
        const int x = ctas[k2];
        const double pi = s_idx * chunk_index_work(begin, k2) / x;
        const double pa0 = s_att * keys * kAttnKeySm / (sms - x), pfl = s_att * keys * kAttnKeyFloor;
        const double pa = pa0 > pfl ? pa0 : pfl;
        s_idx = clampd(s_idx * std::sqrt(1e-3 * t_i / pi), 0.25, 4.0);
        s_att = clampd(s_att * std::sqrt(1e-3 * t_a / pa), 0.25, 4.0);
        const double kj = chunk_attn_keys(begin, j - 1, budget);
        ctas[j] = best_split(s_idx * chunk_index_work(begin, j), s_att * kj * kAttnKeySm, s_att * kj * kAttnKeyFloor,
                             sms);
        return QSA_OK;
    };
    auto run = [&]() -> qsa_status {
        cudaError_t e2 = qsa::launch_kprep(1, 0, L, L, ki, k, k_rot, kblk, freqs, sms, s);
        if (e2 != cudaSuccess) return cuda_fail(e2, "kprep launch");
        if ((e2 = cudaMemsetAsync(stop, 0, sizeof(int), s)) != cudaSuccess) return cuda_fail(e2, "memset");
        if ((e2 = cudaEventRecord(kp[0], s)) != cudaSuccess) return cuda_fail(e2, "event record");
        if ((e2 = cudaStreamWaitEvent(side, kp[0], 0)) != cudaSuccess) return cuda_fail(e2, "stream wait");
        for (int j = 0; j < n; ++j) {
            qsa_status st2 = adapt(j);
            if (st2 != QSA_OK) return st2;
            if ((st2 = enqueue_index(j)) != QSA_OK) return st2;
            if (j > 0 && (st2 = enqueue_attn(j - 1)) != QSA_OK) return st2;
        }
        return enqueue_attn(n - 1);
    };
    st = run();
    cleanup();
    if (st != QSA_OK) return st;
    return ok();
}

qsa_status qsa_kprep_range(const qsa_config *cfg, const qsa_bf16 *ki, const qsa_bf16 *k, qsa_bf16 *k_rot,
                           qsa_bf16 *kblk, int64_t t_begin, int64_t t_end, void *stream) {
    qsa_status st = check_cfg(cfg);
    if (st != QSA_OK) return st;
    if (t_begin < 0 || t_end <= t_begin) return fail(QSA_ERR_INVALID_ARG, "need 0 <= t_begin < t_end");
    if (t_end > kMaxL) return fail(QSA_ERR_UNSUPPORTED, "t_end > %lld", static_cast<long long>(kMaxL));
    REQ_PTR(ki);
    REQ_PTR(kblk);
    if ((k == nullptr) != (k_rot == nullptr))
        return fail(QSA_ERR_INVALID_ARG, "k and k_rot must both be given or both be NULL");
    OPT_PTR(k);
    OPT_PTR(k_rot);
    cudaError_t e = qsa::launch_kprep(1, t_begin, t_end, t_end, ki, k, k_rot, kblk, freqs_of(cfg), sm_count(),
                                      static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kprep launch");
    return ok();
}

size_t qsa_index_topk_cached_workspace_bytes(const qsa_config *cfg, int64_t Lq) {
    if (check_cfg(cfg) != QSA_OK || Lq < 1 || Lq > kMaxL) return 0;
    return align_up(qsa::index_cand_bytes(Lq, sm_count()), 256);
}

size_t qsa_index_topk_tokens_workspace_bytes(const qsa_config *cfg, int64_t L) {
    return qsa_index_topk_cached_workspace_bytes(cfg, L);
}

qsa_status qsa_index_topk_tokens(const qsa_config *cfg, const qsa_bf16 *qi, const qsa_bf16 *w,
                                 const qsa_bf16 *ki, int64_t L, int32_t *idx, float *score, void *ws,
                                 size_t ws_bytes, int32_t *dev_status, void *stream) {
    qsa_status st = check_cfg(cfg);
    if (st != QSA_OK) return st;
    if (L < 1) return fail(QSA_ERR_INVALID_ARG, "L must be >= 1");
    if (L > kMaxL) return fail(QSA_ERR_UNSUPPORTED, "L > %lld", static_cast<long long>(kMaxL));
    REQ_PTR(qi);
    REQ_PTR(w);
    REQ_PTR(ki);
    REQ_PTR(idx);
    OPT_PTR(score);
    REQ_PTR(dev_status);
    const size_t need = qsa_index_topk_tokens_workspace_bytes(cfg, L);
    if (!ws || ws_bytes < need)
        return fail(QSA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, ws_bytes);
    if (!aligned16(ws)) return fail(QSA_ERR_INVALID_ARG, "ws is not 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (cfg->budget_blocks == 1) {
        e = qsa::launch_fill_current_only(0, L, 1, 1, idx, score, s);
        if (e != cudaSuccess) return cuda_fail(e, "selection launch");
        return ok();
    }
    CUtensorMap map_q, map_k;
    st = make_map(&map_q, qi, qsa::kDI, static_cast<uint64_t>(L) * qsa::kHI, 256);
    if (st != QSA_OK) return st;
    st = make_map(&map_k, ki, qsa::kDI, static_cast<uint64_t>(L), 128);  // every token is a unit
    if (st != QSA_OK) return st;
    int *stop = qsa::index_stop_word(ws, qsa::index_cand_bytes(L, sm_count()));
    e = cudaMemsetAsync(stop, 0, sizeof(int), s);
    if (e != cudaSuccess) return cuda_fail(e, "memset");
    e = qsa::launch_index(map_q, map_k, 0, L, 1, cfg->budget_blocks, w, idx, score, nullptr, ws, dev_status,
                          sm_count(), stop, s);
    if (e != cudaSuccess) return cuda_fail(e, "indexer launch");
    return ok();
}

qsa_status qsa_index_topk_cached(const qsa_config *cfg, const qsa_bf16 *qi, const qsa_bf16 *w,
                                 const qsa_bf16 *kblk, int64_t q_offset, int64_t Lq, int32_t *idx,
                                 float *score, void *ws, size_t ws_bytes, int32_t *dev_status,
                                 void *stream) {
    return qsa_index_topk_cached_ctas(cfg, qi, w, kblk, q_offset, Lq, idx, score, 0, ws, ws_bytes, dev_status,
                                      stream);
}

qsa_status qsa_index_topk_cached_ctas(const qsa_config *cfg, const qsa_bf16 *qi, const qsa_bf16 *w,
                                      const qsa_bf16 *kblk, int64_t q_offset, int64_t Lq, int32_t *idx,
                                      float *score, int max_ctas, void *ws, size_t ws_bytes,
                                      int32_t *dev_status, void *stream) {
    qsa_status st = check_cfg(cfg);
    if (st != QSA_OK) return st;
    if (max_ctas < 0) return fail(QSA_ERR_INVALID_ARG, "max_ctas must be >= 0");
    if (Lq < 1) return fail(QSA_ERR_INVALID_ARG, "the number of query rows must be >= 1");
    if (q_offset < 0) return fail(QSA_ERR_INVALID_ARG, "q_offset must be >= 0");
    if (q_offset + Lq > kMaxL) return fail(QSA_ERR_UNSUPPORTED, "more than %lld positions", static_cast<long long>(kMaxL));
    REQ_PTR(qi);
    // w is read one element at a time: a chunk's rows may start at any row
    if (!w || (reinterpret_cast<uintptr_t>(w) & 1u)) return fail(QSA_ERR_INVALID_ARG, "w is NULL or misaligned");
    REQ_PTR(kblk);
    REQ_PTR(idx);
    OPT_PTR(score);
    REQ_PTR(dev_status);
    const size_t need = qsa_index_topk_cached_workspace_bytes(cfg, Lq);
    if (!ws || ws_bytes < need)
        return fail(QSA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, ws_bytes);
    if (!aligned16(ws)) return fail(QSA_ERR_INVALID_ARG, "ws is not 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (cfg->budget_blocks == 1) {
        e = qsa::launch_fill_current_only(q_offset, Lq, qsa::kBlock, 1, idx, score, s);
        if (e != cudaSuccess) return cuda_fail(e, "selection launch");
        return ok();
    }
    CUtensorMap map_q, map_k;
    st = make_map(&map_q, qi, qsa::kDI, static_cast<uint64_t>(Lq) * qsa::kHI, 256);
    if (st != QSA_OK) return st;
    const int64_t nbk = (q_offset + Lq) / qsa::kBlock;
    st = make_map(&map_k, kblk, qsa::kDI, static_cast<uint64_t>(nbk > 0 ? nbk : 1), 128);
    if (st != QSA_OK) return st;
    const int sms = sm_count();
    int *stop = qsa::index_stop_word(ws, qsa::index_cand_bytes(Lq, sms));
    e = cudaMemsetAsync(stop, 0, sizeof(int), s);
    if (e != cudaSuccess) return cuda_fail(e, "memset");
    e = qsa::launch_index(map_q, map_k, q_offset, Lq, qsa::kBlock, cfg->budget_blocks, w, idx, score, nullptr,
                          ws, dev_status, max_ctas > 0 && max_ctas < sms ? max_ctas : sms, stop, s);
    if (e != cudaSuccess) return cuda_fail(e, "indexer launch");
    return ok();
}

size_t qsa_decode_workspace_bytes(const qsa_config *cfg, int batch, int64_t max_ctx) {
    if (check_cfg(cfg) != QSA_OK || batch < 1 || max_ctx < 1 || max_ctx > kMaxDecodeCtx) return 0;
    return qsa::decode_ws_bytes(batch, max_ctx, cfg->budget_blocks, sm_count());
}

qsa_status qsa_sparse_attn_decode(const qsa_config *cfg, int batch, const qsa_bf16 *q,
                                  const qsa_bf16 *qi, const qsa_bf16 *w,
                                  const qsa_bf16 *k_cache, const qsa_bf16 *v_cache,
                                  const qsa_bf16 *kblk_cache, int64_t max_ctx,
                                  const int32_t *seq_lens, qsa_bf16 *out, float *lse,
                                  int32_t *idx_out, void *ws, size_t ws_bytes,
                                  int32_t *dev_status, void *stream) {
    qsa_status st = check_cfg(cfg);
    if (st != QSA_OK) return st;
    if (batch < 1 || batch > 65535) return fail(QSA_ERR_INVALID_ARG, "need 1 <= batch <= 65535");
    if (max_ctx < 1) return fail(QSA_ERR_INVALID_ARG, "max_ctx must be >= 1");
    if (max_ctx > kMaxDecodeCtx)
        return fail(QSA_ERR_UNSUPPORTED, "max_ctx > %lld", static_cast<long long>(kMaxDecodeCtx));
    if (max_ctx % qsa::kBlock) return fail(QSA_ERR_INVALID_ARG, "max_ctx must be a multiple of 4");
    REQ_PTR(q);
    REQ_PTR(qi);
    REQ_PTR(w);
    REQ_PTR(k_cache);
    REQ_PTR(v_cache);
    REQ_PTR(kblk_cache);
    REQ_PTR(seq_lens);
    REQ_PTR(out);
    OPT_PTR(lse);
    OPT_PTR(idx_out);
    REQ_PTR(dev_status);
    const int sms = sm_count();
    const size_t need = qsa::decode_ws_bytes(batch, max_ctx, cfg->budget_blocks, sms);
    // the workspace is checked after every other argument:
    // qsa_sparse_attn_decode_noalloc relies on this order to report argument
    // errors with the statuses of this call
    if (!ws || ws_bytes < need)
        return fail(QSA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, ws_bytes);
    if (!aligned16(ws)) return fail(QSA_ERR_INVALID_ARG, "ws is not 16-byte aligned");

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const qsa::DecodePlan plan = qsa::decode_plan(batch, max_ctx, sms);
    const int budget = cfg->budget_blocks;
    uint8_t *p = static_cast<uint8_t *>(ws);
    auto take = [&](size_t bytes) {
        uint8_t *r = p;
        p += align_up(bytes, 256);
        return r;
    };
    uint8_t *cand_region = take(qsa::decode_index_ws_bytes(batch, max_ctx));
    int32_t *idx_ws = reinterpret_cast<int32_t *>(take(static_cast<size_t>(batch) * budget * 4));
    float *part_o = reinterpret_cast<float *>(take(static_cast<size_t>(batch) * plan.nsplit * qsa::kHQ * qsa::kD * 4));
    float *part_lse = reinterpret_cast<float *>(take(static_cast<size_t>(batch) * plan.nsplit * qsa::kHQ * 4));
    int32_t *idx = idx_out ? idx_out : idx_ws;

    cudaError_t e = qsa::launch_decode_index(batch, max_ctx, plan, qi, w, kblk_cache, seq_lens,
                                             budget, cand_region, idx, dev_status, k_cache, v_cache, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode indexer launch");
    qsa::AttnArgs a{};
    a.q = q;
    a.k = k_cache;
    a.v = v_cache;
    a.seq_stride = max_ctx;
    a.idx = idx;
    a.budget = budget;
    a.seq_lens = seq_lens;
    a.L = 0;
    a.out = out;
    a.lse = lse;
    a.part_o = part_o;
    a.part_lse = part_lse;
    a.nsplit = plan.nsplit;
    a.scale_log2 = scale_log2_of(cfg);
    a.status = dev_status;
    if (use_tc_attention()) {
        CUtensorMap mk, mv;
        qsa_status st2 = make_kv_map(&mk, k_cache, static_cast<uint64_t>(max_ctx), static_cast<uint64_t>(batch));
        if (st2 != QSA_OK) return st2;
        st2 = make_kv_map(&mv, v_cache, static_cast<uint64_t>(max_ctx), static_cast<uint64_t>(batch));
        if (st2 != QSA_OK) return st2;
        e = qsa::launch_attn_decode_tc(a, batch, freqs_of(cfg), mk, mv, s);
    } else {
        e = qsa::launch_attn_decode(a, batch, freqs_of(cfg), s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "decode attention launch");
    if (plan.nsplit > 1) {
        e = qsa::launch_attn_combine(part_o, part_lse, batch, plan.nsplit, out, lse, s);
        if (e != cudaSuccess) return cuda_fail(e, "decode combine launch");
    }
    return ok();
}

}  // extern "C"
