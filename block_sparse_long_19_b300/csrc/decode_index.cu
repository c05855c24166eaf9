// Decode indexer: block scores of one new query per sequence against the
// cached block keys, and the exact selection of the (budget-1) best past
// blocks plus the current block (Qwen3.8-Flash-Next launch post, "Model
// Architecture / Attention: GDN + QSA"; budget from the model card, "Model
// Overview / Qwen Sparse Attention").
//
// The scan streams the block-key cache once (256 B per block; at 1M tokens
// 64 MiB per sequence), so it is bound by HBM bandwidth:
//   * scan kernel: one CTA per (sequence, chunk of blocks); each warp takes
//     16 blocks at a time with 16-byte loads straight into the warp-MMA
//     operand registers (the contraction order inside a 32-dim slice is
//     permuted identically on both operands, which leaves the dot products
//     unchanged), forms s = sum_h w_h max(0, qi_h . kblk) and keeps the chunk's
//     scores in shared memory; a CTA-wide radix select then writes the chunk's
//     exact top-(budget-1) (score desc, block asc) as candidates;
//   * merge kernel: one CTA per sequence selects the final (budget-1) among
//     the chunks' candidates, sorts them by block and appends the current
//     block.
#include "qsa_common.cuh"
#include "qsa_kernels.h"
#include "qsa_select.cuh"

namespace qsa {
namespace dx {

constexpr int SCAN_THREADS = 256;
constexpr int MAX_CHUNK = 16384;
constexpr int MAX_NCHUNK = 47;
constexpr int MERGE_THREADS = 1024;
constexpr int MAX_SEL = kMaxBudget - 1;

// CTA-wide radix step over n items: value(i) -> uint32, pred(i) -> bool.
// Finds a bucket [thr, thr + 2^lo) holding the k-th largest value, looking
// only at the bits below the prefix every valid value shares (candidate
// scores agree on their top bits).  Same contract as the warp version in
// qsa_select.cuh.  ctl: 8 ints of shared memory; all threads must call.
template <int NT, typename Val, typename Pred>
__device__ RadixOut cta_radix(int n, int k, Val value, Pred pred, uint32_t *hist, int *ctl) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t mx = 0u, mn = 0xFFFFFFFFu;
    int nv = 0;
    for (int i = tid; i < n; i += NT)
        if (pred(i)) {
            const uint32_t v = value(i);
            mx = max(mx, v);
            mn = min(mn, v);
            ++nv;
        }
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    mn = __reduce_min_sync(0xFFFFFFFFu, mn);
    nv = __reduce_add_sync(0xFFFFFFFFu, nv);
    if (tid < 3) ctl[tid] = tid == 1 ? static_cast<int>(0xFFFFFFFFu) : 0;
    __syncthreads();
    if (lane == 0) {
        atomicMax(reinterpret_cast<unsigned *>(&ctl[0]), mx);
        atomicMin(reinterpret_cast<unsigned *>(&ctl[1]), mn);
        atomicAdd(&ctl[2], nv);
    }
    __syncthreads();
    mx = static_cast<uint32_t>(ctl[0]);
    mn = static_cast<uint32_t>(ctl[1]);
    nv = ctl[2];
    (void)warp;
    RadixOut r;
    r.krem = k;
    __syncthreads();
    if (mx == mn) {
        r.thr = mx;
        r.eq = nv;
        r.lo = 0;
        return r;
    }
    const int hi = 32 - __clz(mx ^ mn);
    unsigned long long prefix = hi >= 32 ? 0ull : (static_cast<unsigned long long>(mx >> hi) << hi);
    int lo = hi;
    int eq = nv;
    while (lo > 0) {
        const int w = lo >= 8 ? 8 : lo;
        lo -= w;
        const uint32_t dmask = (1u << w) - 1u;
        for (int i = tid; i < 256; i += NT) hist[i] = 0u;
        __syncthreads();
        const unsigned long long want = prefix >> (lo + w);
        for (int i = tid; i < n; i += NT) {
            if (!pred(i)) continue;
            const uint32_t v = value(i);
            if ((static_cast<unsigned long long>(v) >> (lo + w)) == want)
                atomicAdd(&hist[(v >> lo) & dmask], 1u);
        }
        __syncthreads();
        if (tid < 32) {
            uint32_t cnt[8];
            uint32_t sum = 0;
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                cnt[b] = hist[255 - (lane * 8 + b)];
                sum += cnt[b];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += t;
            }
            const uint32_t excl = incl - sum;
            if (excl < static_cast<uint32_t>(r.krem) && static_cast<uint32_t>(r.krem) <= incl) {
                uint32_t acc = excl;
                for (int b = 0; b < 8; ++b) {
                    if (acc + cnt[b] >= static_cast<uint32_t>(r.krem)) {
                        ctl[4] = 255 - (lane * 8 + b);
                        ctl[5] = static_cast<int>(acc);
                        ctl[6] = static_cast<int>(cnt[b]);
                        break;
                    }
                    acc += cnt[b];
                }
            }
        }
        __syncthreads();
        const int digit = ctl[4];
        r.krem -= ctl[5];
        eq = ctl[6];
        prefix |= static_cast<unsigned long long>(digit) << lo;
        __syncthreads();
        if (eq == r.krem) break;
    }
    r.thr = static_cast<uint32_t>(prefix);
    r.eq = eq;
    r.lo = lo;
    return r;
}

// Exact selection of the k best (score desc, block asc) among n items
// given as score(i) (float) and block(i).  Returns the rule: item i is
// selected iff key > t.thr_key, or key == thr_key and ~block >= t.thr_blk
// (thr_blk = 0 selects every item of the bucket when it is exact).
struct SelectRule {
    uint32_t thr_key;
    uint32_t thr_nblk;
    int exact_bucket;  // 1: select key >= thr_key
};
template <int NT, typename Score, typename Block>
__device__ SelectRule cta_select(int n, int k, Score score, Block block, uint32_t *hist, int *ctl) {
    auto kv = [&](int i) { return f2key(score(i)); };
    auto all = [&](int) { return true; };
    const RadixOut r = cta_radix<NT>(n, k, kv, all, hist, ctl);
    SelectRule rule;
    rule.thr_key = r.thr;
    if (r.eq == r.krem) {
        rule.exact_bucket = 1;
        rule.thr_nblk = 0;
        return rule;
    }
    auto nb = [&](int i) { return ~block(i); };
    auto tie = [&](int i) { return kv(i) == r.thr; };
    const RadixOut r2 = cta_radix<NT>(n, r.krem, nb, tie, hist, ctl);
    rule.exact_bucket = 0;
    rule.thr_nblk = r2.thr;
    return rule;
}

__device__ __forceinline__ bool selected(const SelectRule &r, float s, uint32_t b) {
    const uint32_t key = f2key(s);
    if (r.exact_bucket) return key >= r.thr_key;
    return key > r.thr_key || (key == r.thr_key && ~b >= r.thr_nblk);
}

struct ScanParams {
    const uint16_t *qi;        // [B, 4, 128]
    const uint16_t *w;         // [B, 4]
    const uint16_t *kblk;      // [B, max_ctx/4, 128]
    const int32_t *seq_lens;   // [B]
    int64_t max_ctx;
    int64_t chunk;
    int nchunk;
    int k_sel;
    uint2 *cand;               // [B, nchunk, k_sel]
    int32_t *cnt;              // [B, nchunk]
    uint32_t *thr;             // [B] running max of the chunks' (budget-1)-th best key
    int32_t *status;
};

__global__ void __launch_bounds__(SCAN_THREADS) scan_kernel(ScanParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    float *sc = reinterpret_cast<float *>(smem);
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + p.chunk * 4);  // dynamic size: chunk*4 + 256*4 + 32
    int *ctl = reinterpret_cast<int *>(hist + 256);

    const int s = blockIdx.y;
    const int ch = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t T = p.seq_lens[s];
    int32_t *cnt_out = p.cnt + static_cast<int64_t>(s) * p.nchunk + ch;
    if (T < 1 || T > p.max_ctx) {
        if (threadIdx.x == 0) {
            report(p.status, QSA_ERR_DEVICE_CHECK);
            *cnt_out = 0;
        }
        return;
    }
    const int64_t c = (T - 1) / kBlock;  // past blocks 0..c-1
    const int64_t b0 = static_cast<int64_t>(ch) * p.chunk;
    int64_t b1 = b0 + p.chunk;
    if (b1 > c) b1 = c;
    if (b0 >= b1) {
        if (threadIdx.x == 0) *cnt_out = 0;
        return;
    }
    const int n = static_cast<int>(b1 - b0);

    // B operand: qi^T, columns = heads (4 live of 8), loaded once
    const int qd = lane & 3, hr = lane >> 2;
    uint4 bq[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        bq[kk] = hr < kHI ? *reinterpret_cast<const uint4 *>(
                                p.qi + (static_cast<int64_t>(s) * kHI + hr) * kDI + kk * 32 + qd * 8)
                          : make_uint4(0, 0, 0, 0);
    float w0 = 0.f, w1 = 0.f;
    if (qd < 2) {
        w0 = __uint_as_float(static_cast<uint32_t>(p.w[s * kHI + 2 * qd]) << 16);
        w1 = __uint_as_float(static_cast<uint32_t>(p.w[s * kHI + 2 * qd + 1]) << 16);
    }
    const uint16_t *kb = p.kblk + static_cast<int64_t>(s) * (p.max_ctx / kBlock) * kDI;

    for (int mt = warp; mt * 16 < n; mt += SCAN_THREADS / 32) {
        const int64_t ra = b0 + mt * 16 + hr;
        const int64_t rb = ra + 8;
        const int64_t la = ra < b1 ? ra : b1 - 1;
        const int64_t lb = rb < b1 ? rb : b1 - 1;
        uint4 ua[4], ub[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            ua[kk] = __ldcs(reinterpret_cast<const uint4 *>(kb + la * kDI + kk * 32 + qd * 8));
            ub[kk] = __ldcs(reinterpret_cast<const uint4 *>(kb + lb * kDI + kk * 32 + qd * 8));
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            mma_bf16_16816(acc, ua[kk].x, ub[kk].x, ua[kk].y, ub[kk].y, bq[kk].x, bq[kk].y);
            mma_bf16_16816(acc, ua[kk].z, ub[kk].z, ua[kk].w, ub[kk].w, bq[kk].z, bq[kk].w);
        }
        float pa = w0 * fmaxf(acc[0], 0.f) + w1 * fmaxf(acc[1], 0.f);  // row hr
        float pb = w0 * fmaxf(acc[2], 0.f) + w1 * fmaxf(acc[3], 0.f);  // row hr + 8
        pa += __shfl_xor_sync(0xFFFFFFFFu, pa, 1);
        pb += __shfl_xor_sync(0xFFFFFFFFu, pb, 1);
        if (qd == 0) {
            if (ra < b1) sc[ra - b0] = pa + 0.0f;
            if (rb < b1) sc[rb - b0] = pb + 0.0f;
        }
    }
    __syncthreads();

    uint2 *out = p.cand + (static_cast<int64_t>(s) * p.nchunk + ch) * p.k_sel;
    if (n <= p.k_sel) {
        for (int i = threadIdx.x; i < n; i += SCAN_THREADS)
            out[i] = make_uint2(__float_as_uint(sc[i]), static_cast<uint32_t>(b0 + i));
        if (threadIdx.x == 0) *cnt_out = n;
        return;
    }
    const SelectRule rule = cta_select<SCAN_THREADS>(
        n, p.k_sel, [&](int i) { return sc[i]; },
        [&](int i) { return static_cast<uint32_t>(b0 + i); }, hist, ctl);
    // This chunk holds budget-1 blocks whose keys are >= rule.thr_key, so the
    // sequence's (budget-1)-th best key is >= it too: publish it.  Candidates
    // below the largest bound published so far can never be selected.
    if (threadIdx.x == 0) {
        const uint32_t old = atomicMax(&p.thr[s], rule.thr_key);
        ctl[7] = static_cast<int>(max(old, rule.thr_key));
        ctl[3] = 0;
    }
    __syncthreads();
    const uint32_t bound = static_cast<uint32_t>(ctl[7]);
    for (int i = threadIdx.x; i < n; i += SCAN_THREADS) {
        if (selected(rule, sc[i], static_cast<uint32_t>(b0 + i)) && f2key(sc[i]) >= bound) {
            const int pos = atomicAdd(&ctl[3], 1);
            if (pos < p.k_sel)
                out[pos] = make_uint2(__float_as_uint(sc[i]), static_cast<uint32_t>(b0 + i));
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (ctl[3] > p.k_sel) report(p.status, QSA_ERR_DEVICE_CHECK);
        *cnt_out = min(ctl[3], p.k_sel);
    }
}

struct MergeParams {
    const int32_t *seq_lens;
    int64_t max_ctx;
    int nchunk;
    int k_sel;
    int budget;
    const uint2 *cand;
    const int32_t *cnt;
    const uint32_t *thr;  // [B] lower bound of the (budget-1)-th best key (null: none)
    int32_t *idx;   // [B, budget]
    int32_t *status;
};

__global__ void __launch_bounds__(MERGE_THREADS) merge_kernel(MergeParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint2 *items = reinterpret_cast<uint2 *>(smem);
    const int cap = MAX_NCHUNK * MAX_SEL;
    unsigned long long *sortb = reinterpret_cast<unsigned long long *>(items + cap);
    uint32_t *hist = reinterpret_cast<uint32_t *>(sortb + kMaxBudget);
    int *ctl = reinterpret_cast<int *>(hist + 256);

    const int s = blockIdx.x;
    const int64_t T = p.seq_lens[s];
    int32_t *row = p.idx + static_cast<int64_t>(s) * p.budget;
    if (T < 1 || T > p.max_ctx) {
        if (threadIdx.x == 0) report(p.status, QSA_ERR_DEVICE_CHECK);
        for (int i = threadIdx.x; i < p.budget; i += MERGE_THREADS) row[i] = -1;
        return;
    }
    const int64_t c = (T - 1) / kBlock;
    // every warp takes whole chunks: all of a chunk's candidate loads in
    // flight at once, the ones at or above the bound appended with one
    // shared atomic per warp
    if (threadIdx.x == 0) ctl[3] = 0;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned ltmask = (1u << lane) - 1u;
    const uint32_t bound = p.thr ? p.thr[s] : 0u;
    constexpr int PER_LANE = (MAX_SEL + 31) / 32;
    for (int ch = warp; ch < p.nchunk; ch += MERGE_THREADS / 32) {
        const int cnt = p.k_sel > 0 ? min(p.cnt[static_cast<int64_t>(s) * p.nchunk + ch], p.k_sel) : 0;
        const uint2 *src = p.cand + (static_cast<int64_t>(s) * p.nchunk + ch) * p.k_sel;
        uint2 it[PER_LANE];
#pragma unroll
        for (int u = 0; u < PER_LANE; ++u) {
            const int i = u * 32 + lane;
            it[u] = i < cnt ? src[i] : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < PER_LANE; ++u) {
            if (u * 32 >= cnt) break;
            const bool ok = u * 32 + lane < cnt && f2key(__uint_as_float(it[u].x)) >= bound;
            const unsigned ball = __ballot_sync(0xFFFFFFFFu, ok);
            if (!ball) continue;
            int base = 0;
            if (lane == 0) base = atomicAdd(&ctl[3], __popc(ball));
            base = __shfl_sync(0xFFFFFFFFu, base, 0);
            const int pos = base + __popc(ball & ltmask);
            if (ok && pos < cap) items[pos] = it[u];
        }
    }
    __syncthreads();
    const int n = min(ctl[3], cap);
    __syncthreads();
    SelectRule rule{0u, 0u, 1};
    if (n > p.k_sel)
        rule = cta_select<MERGE_THREADS>(
            n, p.k_sel, [&](int i) { return __uint_as_float(items[i].x); },
            [&](int i) { return items[i].y; }, hist, ctl);
    if (threadIdx.x == 0) ctl[3] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += MERGE_THREADS) {
        const int i = i0 + threadIdx.x;
        const bool sel = i < n && (n <= p.k_sel || selected(rule, __uint_as_float(items[i].x), items[i].y));
        const unsigned ball = __ballot_sync(0xFFFFFFFFu, sel);
        if (!ball) continue;
        int base = 0;
        if (lane == 0) base = atomicAdd(&ctl[3], __popc(ball));
        base = __shfl_sync(0xFFFFFFFFu, base, 0);
        const int pos = base + __popc(ball & ltmask);
        if (sel && pos < kMaxBudget) sortb[pos] = (static_cast<unsigned long long>(items[i].y) << 32) | items[i].x;
    }
    __syncthreads();
    // order by block: blocks are distinct, so an item's place is the number
    // of smaller blocks (every thread scans the list with broadcast reads)
    const int m = min(ctl[3], kMaxBudget);
    for (int i = threadIdx.x; i < m; i += MERGE_THREADS) {
        const uint32_t bi = static_cast<uint32_t>(sortb[i] >> 32);
        int rank = 0;
        for (int j = 0; j < m; ++j) rank += static_cast<uint32_t>(sortb[j] >> 32) < bi;
        if (rank < p.budget) row[rank] = static_cast<int32_t>(bi);
    }
    for (int i = m + threadIdx.x; i < p.budget; i += MERGE_THREADS)
        row[i] = i == m ? static_cast<int32_t>(c) : -1;
}

}  // namespace dx

DecodePlan decode_plan(int batch, int64_t max_ctx, int sms) {
    DecodePlan pl;
    const int64_t cmax = (max_ctx - 1) / kBlock;
    int64_t target = (static_cast<int64_t>(batch) * cmax + static_cast<int64_t>(sms) * 4 - 1) /
                     (static_cast<int64_t>(sms) * 4);
    int64_t ch = ((target + 255) / 256) * 256;
    if (ch < 1024) ch = 1024;
    if (ch > dx::MAX_CHUNK) ch = dx::MAX_CHUNK;
    int64_t nchunk = cmax > 0 ? (cmax + ch - 1) / ch : 1;
    if (nchunk > dx::MAX_NCHUNK) {
        ch = (((cmax + dx::MAX_NCHUNK - 1) / dx::MAX_NCHUNK + 255) / 256) * 256;
        nchunk = (cmax + ch - 1) / ch;
    }
    pl.chunk = ch;
    pl.nchunk = static_cast<int>(nchunk < 1 ? 1 : nchunk);
    int nsplit = (2 * sms + batch - 1) / batch;
    if (nsplit > 16) nsplit = 16;
    if (nsplit < 1) nsplit = 1;
    pl.nsplit = nsplit;
    return pl;
}

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

size_t decode_ws_bytes(int batch, int64_t max_ctx, int budget, int sms) {
    const DecodePlan pl = decode_plan(batch, max_ctx, sms);
    const int k_sel = budget - 1 > 0 ? budget - 1 : 1;
    size_t b = 0;
    b += align256(static_cast<size_t>(batch) * pl.nchunk * k_sel * sizeof(uint2));   // cand
    b += align256(static_cast<size_t>(batch) * pl.nchunk * sizeof(int32_t));         // cnt
    b += align256(static_cast<size_t>(batch) * sizeof(uint32_t));                    // thr
    b += align256(static_cast<size_t>(batch) * budget * sizeof(int32_t));            // idx
    b += align256(static_cast<size_t>(batch) * pl.nsplit * kHQ * kD * sizeof(float)); // part_o
    b += align256(static_cast<size_t>(batch) * pl.nsplit * kHQ * sizeof(float));      // part_lse
    return b;
}

cudaError_t launch_decode_index(int batch, int64_t max_ctx, const DecodePlan &plan,
                                const uint16_t *qi, const uint16_t *w, const uint16_t *kblk,
                                const int32_t *seq_lens, int budget, void *ws, int32_t *idx_out,
                                int32_t *status, cudaStream_t stream) {
    const int k_sel = budget - 1;
    uint8_t *base = static_cast<uint8_t *>(ws);
    const int k_alloc = k_sel > 0 ? k_sel : 1;
    uint2 *cand = reinterpret_cast<uint2 *>(base);
    base += align256(static_cast<size_t>(batch) * plan.nchunk * k_alloc * sizeof(uint2));
    int32_t *cnt = reinterpret_cast<int32_t *>(base);
    base += align256(static_cast<size_t>(batch) * plan.nchunk * sizeof(int32_t));
    uint32_t *thr = reinterpret_cast<uint32_t *>(base);
    cudaError_t e;
    if (k_sel > 0) {
        e = cudaMemsetAsync(thr, 0, static_cast<size_t>(batch) * sizeof(uint32_t), stream);
        if (e != cudaSuccess) return e;
        dx::ScanParams sp;
        sp.qi = qi;
        sp.w = w;
        sp.kblk = kblk;
        sp.seq_lens = seq_lens;
        sp.max_ctx = max_ctx;
        sp.chunk = plan.chunk;
        sp.nchunk = plan.nchunk;
        sp.k_sel = k_sel;
        sp.cand = cand;
        sp.cnt = cnt;
        sp.thr = thr;
        sp.status = status;
        const int smem = static_cast<int>(plan.chunk * 4 + 256 * 4 + 32);
        e = cudaFuncSetAttribute(dx::scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        dim3 grid(plan.nchunk, batch);
        dx::scan_kernel<<<grid, dx::SCAN_THREADS, smem, stream>>>(sp);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    dx::MergeParams mp;
    mp.seq_lens = seq_lens;
    mp.max_ctx = max_ctx;
    mp.nchunk = plan.nchunk;
    mp.k_sel = k_sel;
    mp.budget = budget;
    mp.cand = cand;
    mp.cnt = cnt;
    mp.thr = k_sel > 0 ? thr : nullptr;
    mp.idx = idx_out;
    mp.status = status;
    const int smem = dx::MAX_NCHUNK * dx::MAX_SEL * 8 + kMaxBudget * 8 + 256 * 4 + 8 * 4 +
                     (dx::MAX_NCHUNK + 1) * 4;
    e = cudaFuncSetAttribute(dx::merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dx::merge_kernel<<<batch, dx::MERGE_THREADS, smem, stream>>>(mp);
    return cudaGetLastError();
}

}  // namespace qsa
