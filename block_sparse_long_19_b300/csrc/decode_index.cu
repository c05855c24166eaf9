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
//     unchanged) and forms s = sum_h w_h max(0, qi_h . kblk).  The chunk's
//     scores go to the workspace (L2-resident: 4 B per block), and the
//     chunk's kc-th best score with kc = ceil((budget-1) / (chunks - 1)) is
//     found: every full chunk holds kc blocks at or above its own value, so
//     the smallest value over the chunks is a lower bound of the sequence's
//     (budget-1)-th best score.  Where kc is small (long contexts: 15 at
//     1M tokens) each lane keeps its best keys in registers while the chunk
//     streams and the kc-th best comes from the warps' merged lists, so no
//     pass over the chunk's scores follows the stream; with more chunks'
//     worth of kc each warp bounds its own blocks the same way (kw-th best),
//     and only with few chunks does a CTA radix step run over the scores;
//   * filter kernel: every block whose score reaches that bound becomes a
//     candidate (on i.i.d. scores about twice the budget survive); at small
//     batch the candidates' K and V rows are also prefetched into L2 for the
//     decode attention, while HBM is otherwise idle;
//   * merge kernel: one CTA per sequence selects the exact (budget-1) best
//     candidates (score desc, block asc), sorts them by block and appends the
//     current block.  If ties leave more candidates than the candidate area
//     holds, it selects over all of the sequence's scores instead.
#include <cmath>

#include "qsa_common.cuh"
#include "qsa_kernels.h"
#include "qsa_select.cuh"

namespace qsa {
namespace dx {

constexpr int SCAN_THREADS = 256;
constexpr int MAX_CHUNK = 16384;
constexpr int MAX_NCHUNK = 256;  // scan CTAs per sequence
constexpr int KW_MAX = 16;       // best scores kept per lane (and per warp) for the chunk bound
constexpr int MERGE_THREADS = 256;
constexpr int MERGE_SPEC = 8;  // candidates per merge thread loaded before their count is known
constexpr int FILTER_THREADS = 256;
constexpr int FILTER_PER_THREAD = 8;
constexpr int CAND_CAP = 8192;  // filtered candidates kept per sequence
static_assert(MERGE_SPEC * MERGE_THREADS <= CAND_CAP, "speculative loads stay in the candidate area");
constexpr int CCOUNT_STRIDE = 32;  // ints between two sequences' candidate counters (128 B)
constexpr int64_t kPrefetchL2Bytes = int64_t(72) << 20;  // L2 budget of the filter's K/V prefetch

// CTA-wide radix step over n items: value(i) -> uint32, pred(i) -> bool.
// Finds a bucket [thr, thr + 2^lo) holding the k-th largest value, looking
// only at the bits below the prefix every valid value shares (candidate
// scores agree on their top bits), with at most max_passes 8-bit digit
// passes (4 passes reach every bit: the bucket is then exact).  Same
// contract as the warp version in qsa_select.cuh.  ctl: 8 ints of shared
// memory; all threads must call.
template <int NT, typename Val, typename Pred>
__device__ RadixOut cta_radix(int n, int k, Val value, Pred pred, uint32_t *hist, int *ctl, int max_passes = 4) {
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
    for (int pass = 0; pass < max_passes && lo > 0; ++pass) {
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

// How the scan bounds a sequence with c past blocks (see scan_kernel), and
// where the bound slots that the filter reduces sit: chunk and radix modes
// fill slot 0 of each chunk, warp mode the slots of every warp.
constexpr int SCAN_WARPS = SCAN_THREADS / 32;
struct BoundMode {
    int64_t nch;     // chunks of the sequence
    int kc, kw;      // ranks of the chunk and of the warp bounds
    bool chunk_mode, warp_mode;
};
__device__ __forceinline__ BoundMode bound_mode(int64_t c, int64_t chunk, int k_sel) {
    // 32-bit arithmetic: c < 2^20 blocks per sequence, chunk <= MAX_CHUNK
    BoundMode m;
    const int ci = static_cast<int>(c), chi = static_cast<int>(chunk);
    const int nch = (ci + chi - 1) / chi;
    m.nch = nch;
    m.kc = nch == 1 ? k_sel : (k_sel + nch - 2) / (nch - 1);
    const int wfull = (nch - 1) * SCAN_WARPS;  // warps of full chunks: >= chunk / 8 >= 128 scores each
    m.kw = wfull > 1 ? (k_sel + wfull - 2) / (wfull - 1) : KW_MAX + 1;
    const bool sel_needed = c > k_sel && m.nch > 1;
    m.chunk_mode = sel_needed && m.kc <= KW_MAX;
    m.warp_mode = sel_needed && !m.chunk_mode && m.kw <= KW_MAX;
    return m;
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
    float *scores;             // [B, max_ctx/4]
    uint32_t *lb;              // [B, nchunk, SCAN_THREADS / 32] bound keys of the chunks or their warps (0xFFFFFFFF: none)
    int32_t *ccount;           // [B x CCOUNT_STRIDE] candidate counters, zeroed here for the filter
    int32_t *status;
};

__global__ void __launch_bounds__(SCAN_THREADS, 2) scan_kernel(ScanParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    float *sc = reinterpret_cast<float *>(smem);
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + p.chunk * 4);  // dynamic size: chunk*4 + 256*4 + 32
    int *ctl = reinterpret_cast<int *>(hist + 256);

    pdl_trigger();
    const int s = blockIdx.y;
    const int ch = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t T = p.seq_lens[s];
    constexpr int NW = SCAN_THREADS / 32;
    // the chunk's bound slots, one per warp: lane 0 of warp w clears slot w
    // here and is the only thread that writes it below
    uint32_t *lb_out = p.lb + (static_cast<int64_t>(s) * p.nchunk + ch) * NW;
    if (lane == 0) lb_out[warp] = 0xFFFFFFFFu;
    if (threadIdx.x == 0 && ch == 0) p.ccount[static_cast<int64_t>(s) * CCOUNT_STRIDE] = 0;
    if (T < 1 || T > p.max_ctx) {
        if (threadIdx.x == 0) report(p.status, QSA_ERR_DEVICE_CHECK);
        return;
    }
    const int64_t c = (T - 1) / kBlock;  // past blocks 0..c-1
    const int64_t b0 = static_cast<int64_t>(ch) * p.chunk;
    int64_t b1 = b0 + p.chunk;
    if (b1 > c) b1 = c;
    if (b0 >= b1) return;
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
    // The sequence's bound is the smallest of per-chunk (or per-warp) values
    // that each have enough scores at or above them:
    //  * chunk (kc <= KW_MAX): the chunk's kc-th best key with kc = ceil(
    //    (budget-1) / (chunks-1)), merged from the warps' best kc keys (each
    //    lane keeps its best KW_MAX while the chunk streams, so no pass over
    //    the chunk's scores follows the stream);
    //  * warp (kw <= KW_MAX): each warp's kw-th best with kw = ceil((budget-1)
    //    / (warps of full chunks - 1)), looser but with no merge across warps;
    //  * otherwise the chunk's kc-th best by a CTA radix after the stream.
    const BoundMode bm = bound_mode(c, p.chunk, p.k_sel);
    const int kc = bm.kc, kw = bm.kw;
    const bool chunk_mode = bm.chunk_mode, warp_mode = bm.warp_mode;
    const bool keep_top = chunk_mode || warp_mode;
    uint32_t top[KW_MAX];  // this lane's best keys, descending (lanes with qd == 0 hold scores)
#pragma unroll
    for (int j = 0; j < KW_MAX; ++j) top[j] = 0u;
    int nmine = 0;

    // two 16-block tiles per warp and iteration: all 16 loads of a lane in
    // flight before the first MMA
    for (int mt0 = warp; mt0 * 16 < n; mt0 += 2 * NW) {
        uint4 ua[2][4], ub[2][4];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int64_t ra = b0 + (mt0 + h2 * NW) * 16 + hr;
            const int64_t la = ra < b1 ? ra : b1 - 1;
            const int64_t lb = ra + 8 < b1 ? ra + 8 : b1 - 1;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                ua[h2][kk] = __ldcs(reinterpret_cast<const uint4 *>(kb + la * kDI + kk * 32 + qd * 8));
                ub[h2][kk] = __ldcs(reinterpret_cast<const uint4 *>(kb + lb * kDI + kk * 32 + qd * 8));
            }
        }
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int64_t ra = b0 + (mt0 + h2 * NW) * 16 + hr;
            const int64_t rb = ra + 8;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                mma_bf16_16816(acc, ua[h2][kk].x, ub[h2][kk].x, ua[h2][kk].y, ub[h2][kk].y, bq[kk].x, bq[kk].y);
                mma_bf16_16816(acc, ua[h2][kk].z, ub[h2][kk].z, ua[h2][kk].w, ub[h2][kk].w, bq[kk].z, bq[kk].w);
            }
            float pa = w0 * fmaxf(acc[0], 0.f) + w1 * fmaxf(acc[1], 0.f);  // row hr
            float pb = w0 * fmaxf(acc[2], 0.f) + w1 * fmaxf(acc[3], 0.f);  // row hr + 8
            pa += __shfl_xor_sync(0xFFFFFFFFu, pa, 1);
            pb += __shfl_xor_sync(0xFFFFFFFFu, pb, 1);
            if (qd == 0) {
                if (ra < b1) sc[ra - b0] = pa + 0.0f;
                if (rb < b1) sc[rb - b0] = pb + 0.0f;
                if (keep_top) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        if ((e == 0 ? ra : rb) >= b1) continue;
                        uint32_t v = f2key((e == 0 ? pa : pb) + 0.0f);
                        ++nmine;
#pragma unroll
                        for (int j = 0; j < KW_MAX; ++j) {  // insert, keeping top[] descending
                            const uint32_t hi = max(top[j], v);
                            v = min(top[j], v);
                            top[j] = hi;
                        }
                    }
                }
            }
        }
    }
    uint32_t *wtop = hist;  // [NW][KW_MAX] the warps' best keys, descending
    int *wcnt = ctl;        // [NW] valid entries of each warp's list
    if (keep_top) {
        // the warp's best keys: the largest head of the lanes' lists, taken out
        // one copy at a time (equal keys count separately); kc of them for the
        // chunk bound, kw for the warp's own
        const int want = chunk_mode ? kc : kw;
        const int nlist = min(nmine, KW_MAX);
        int taken = 0;  // entries this lane gave up (its list shifts up by one each time)
        int nw = 0;     // entries of the warp's list (warp-uniform)
        uint32_t last = 0u;
#pragma unroll 1
        for (int r = 0; r < want; ++r) {
            const bool live = qd == 0 && taken < nlist;
            if (!__any_sync(0xFFFFFFFFu, live)) break;
            const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, live ? top[0] : 0u);
            const unsigned who = __ballot_sync(0xFFFFFFFFu, live && top[0] == mx);
            if (lane == __ffs(who) - 1) {
#pragma unroll
                for (int j = 0; j + 1 < KW_MAX; ++j) top[j] = top[j + 1];
                ++taken;
            }
            if (lane == 0) wtop[warp * KW_MAX + r] = mx;
            last = mx;
            ++nw;
        }
        if (lane == 0) {
            wcnt[warp] = nw;
            if (warp_mode && nw == kw) lb_out[warp] = last;  // at least kw of the warp's keys are >= last
        }
    }
    __syncthreads();

    float *srow = p.scores + static_cast<int64_t>(s) * (p.max_ctx / kBlock);
    for (int i = threadIdx.x; i < n; i += SCAN_THREADS) srow[b0 + i] = sc[i];
    if (c <= p.k_sel || warp_mode) return;  // every past block is selected, or the warps bound
    if (n < kc) return;  // a short last chunk: the full chunks already cover the bound
    if (chunk_mode) {
        // the kc-th best of the warps' lists (lanes 0..NW-1 each walk one list)
        if (warp == 0) {
            const int nl = lane < NW ? wcnt[lane] : 0;
            int hd = 0;
            uint32_t kth = 0u;
            int got = 0;
#pragma unroll 1
            for (int r = 0; r < kc; ++r) {
                const bool live = hd < nl;
                if (!__any_sync(0xFFFFFFFFu, live)) break;
                const uint32_t head = live ? wtop[lane * KW_MAX + hd] : 0u;
                const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, head);
                const unsigned who = __ballot_sync(0xFFFFFFFFu, live && head == mx);
                if (lane == __ffs(who) - 1) ++hd;
                kth = mx;
                ++got;
            }
            // got < kc only if the lists hold fewer than kc keys: no bound then
            if (lane == 0 && got == kc) lb_out[0] = kth;
        }
        return;
    }
    // two digit passes: the bucket floor is a lower bound of the kc-th best
    // key within about 2^-8 of it (16 bits below the keys' shared prefix),
    // and the passes that would make it exact are not spent
    const RadixOut r = cta_radix<SCAN_THREADS>(
        n, kc, [&](int i) { return f2key(sc[i]); }, [&](int) { return true; }, hist, ctl, 2);
    // at least kc of this chunk's keys are >= r.thr
    if (threadIdx.x == 0) lb_out[0] = r.thr;
}

struct MergeParams {
    const int32_t *seq_lens;
    int64_t max_ctx;
    int k_sel;
    int budget;
    const float *scores;    // [B, max_ctx/4] (used when the candidates overflowed)
    const uint2 *cand;      // [B, CAND_CAP]
    const int32_t *ccount;  // [B x CCOUNT_STRIDE]
    int32_t *idx;           // [B, budget]
    int32_t *status;
};

// The selection row of sequence s whose candidates are complete: the exact
// (budget-1) best candidates (score desc, block asc), sorted by block, then
// the current block.  Candidates up to items_cap are staged in shared
// memory (`items`), more are read from the candidate area in L2, and if ties
// flooded that area the selection runs over all of the sequence's scores.
// sortb: 1024 words; hist: 256 words; ctl: 8 ints.  All NT threads call.
template <int NT>
__device__ void merge_row(const MergeParams &p, int s, int64_t c, uint2 *items, int items_cap, uint32_t *sortb,
                          uint32_t *hist, int *ctl) {
    int32_t *row = p.idx + static_cast<int64_t>(s) * p.budget;
    const int lane = threadIdx.x & 31;
    const unsigned ltmask = (1u << lane) - 1u;
    // the first MERGE_SPEC * NT candidates are loaded together with their
    // count (one round trip to L2 instead of two); entries past the count are
    // loaded but not used (the area holds CAND_CAP entries per sequence)
    const uint2 *src = p.cand + static_cast<int64_t>(s) * CAND_CAP;
    uint2 pre[MERGE_SPEC];
#pragma unroll
    for (int k = 0; k < MERGE_SPEC; ++k) pre[k] = __ldcg(src + threadIdx.x + k * NT);
    const int nc = __ldcg(p.ccount + static_cast<int64_t>(s) * CCOUNT_STRIDE);
    const bool direct = nc > CAND_CAP;  // ties flooded the candidate area
    const bool staged = !direct && nc <= items_cap;
    const int n = direct ? static_cast<int>(c) : nc;
    const float *srow = p.scores + static_cast<int64_t>(s) * (p.max_ctx / kBlock);
    if (staged) {
#pragma unroll
        for (int k = 0; k < MERGE_SPEC; ++k)
            if (threadIdx.x + k * NT < n) items[threadIdx.x + k * NT] = pre[k];
#pragma unroll 4
        for (int i = threadIdx.x + MERGE_SPEC * NT; i < n; i += NT) items[i] = __ldcg(src + i);
    }
    __syncthreads();
    auto score = [&](int i) {
        return direct ? __ldcg(srow + i) : __uint_as_float(staged ? items[i].x : __ldcg(&src[i].x));
    };
    auto block = [&](int i) { return direct ? static_cast<uint32_t>(i) : (staged ? items[i].y : __ldcg(&src[i].y)); };
    SelectRule rule{0u, 0u, 1};
    if (n > p.k_sel) rule = cta_select<NT>(n, p.k_sel, score, block, hist, ctl);
    if (threadIdx.x == 0) ctl[3] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += NT) {
        const int i = i0 + threadIdx.x;
        float sv = 0.f;
        uint32_t bv = 0u;
        if (i < n) {
            sv = score(i);
            bv = block(i);
        }
        const bool sel = i < n && (n <= p.k_sel || selected(rule, sv, bv));
        const unsigned ball = __ballot_sync(0xFFFFFFFFu, sel);
        if (!ball) continue;
        int pos0 = 0;
        if (lane == 0) pos0 = atomicAdd(&ctl[3], __popc(ball));
        pos0 = __shfl_sync(0xFFFFFFFFu, pos0, 0);
        const int pos = pos0 + __popc(ball & ltmask);
        if (sel && pos < kMaxBudget) sortb[512 + pos] = bv;
    }
    __syncthreads();
    const int m = min(ctl[3], p.k_sel);
    if (threadIdx.x == 0 && ctl[3] != p.k_sel) report(p.status, QSA_ERR_DEVICE_CHECK);
    // order by block (blocks are distinct): a bitonic sort of 512 keys by the
    // first four warps, padded with the largest key
    if (threadIdx.x < 128) {
        uint32_t v[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int e = 4 * threadIdx.x + r;
            v[r] = e < m ? sortb[512 + e] : 0xFFFFFFFFu;
        }
        group_sort512(v, sortb, threadIdx.x, 1);
#if QSA_DEBUG_CHECKS
#pragma unroll
        for (int r = 0; r < 4; ++r)
            if (4 * threadIdx.x + r < m)
                debug_check(p.status, v[r] < static_cast<uint64_t>(c) && (r == 0 || v[r - 1] < v[r]));
#endif
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int e = 4 * threadIdx.x + r;
            if (e < m && e < p.budget) row[e] = static_cast<int32_t>(v[r]);
        }
    }
    for (int i = m + threadIdx.x; i < p.budget; i += NT) row[i] = i == m ? static_cast<int32_t>(c) : -1;
}

// A row that needs no selection: an invalid length (all -1), or every past
// block (none for budget 1) and then the current block.  Returns true for
// such a row, which it writes if `write` is set.
template <int NT>
__device__ bool trivial_row(const MergeParams &p, int s, bool write) {
    const int64_t T = p.seq_lens[s];
    int32_t *row = p.idx + static_cast<int64_t>(s) * p.budget;
    if (T < 1 || T > p.max_ctx) {
        if (write) {
            if (threadIdx.x == 0) report(p.status, QSA_ERR_DEVICE_CHECK);
            for (int i = threadIdx.x; i < p.budget; i += NT) row[i] = -1;
        }
        return true;
    }
    const int64_t c = (T - 1) / kBlock;
    if (c <= p.k_sel || p.k_sel <= 0) {
        const int64_t np = p.k_sel <= 0 ? 0 : c;
        if (write)
            for (int i = threadIdx.x; i < p.budget; i += NT)
                row[i] = i < np ? i : (i == np ? static_cast<int32_t>(c) : -1);
        return true;
    }
    return false;
}

struct FilterParams {
    MergeParams m;           // lengths, budget and scores of the sequences
    const uint32_t *lb;      // [B, nchunk, SCAN_THREADS / 32]
    int nchunk;
    int64_t chunk;           // blocks per scan chunk
    uint2 *cand;             // [B, CAND_CAP] {score bits, block}
    int32_t *ccount;         // [B x CCOUNT_STRIDE] candidates reserved
    const uint16_t *kpre;    // [B, max_ctx, 2, 256] K cache to prefetch into L2 (or null)
    const uint16_t *vpre;    // [B, max_ctx, 2, 256] V cache
    int pre_cap;             // candidates prefetched per sequence at most
};

// Candidates: the past blocks whose score key reaches the sequence's bound.
// One global atomic per CTA reserves the CTA's range of the candidate area
// (per-warp atomics from every CTA would queue up at the counter's L2 slice);
// the sequences' counters sit 128 bytes apart, on cache lines of their own.
__global__ void __launch_bounds__(FILTER_THREADS) filter_kernel(FilterParams p) {
    __shared__ int s_warp[FILTER_THREADS / 32 + 1];
    pdl_trigger();
    // the sequence length is an input of the step (no earlier kernel writes
    // it): it is read while the scan finishes
    const int s = blockIdx.y;
    if (trivial_row<FILTER_THREADS>(p.m, s, false)) return;  // the merge writes that row
    const int64_t c = (p.m.seq_lens[s] - 1) / kBlock;
    pdl_wait();  // scores and bounds of the scan
    const float *srow = p.m.scores + static_cast<int64_t>(s) * (p.m.max_ctx / kBlock);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned ltmask = (1u << lane) - 1u;
    // this CTA's scores: all loads in flight at once, before the bound is known
    const int64_t base = static_cast<int64_t>(blockIdx.x) * FILTER_THREADS * FILTER_PER_THREAD;
    float v[FILTER_PER_THREAD];
#pragma unroll
    for (int u = 0; u < FILTER_PER_THREAD; ++u) {
        const int64_t b = base + u * FILTER_THREADS + threadIdx.x;
        v[u] = b < c ? __ldcg(srow + b) : -INFINITY;
    }
    // the bound: the smallest chunk or warp bound (slots that bound nothing
    // hold 0xFFFFFFFF); every warp reduces the slots itself
    const uint32_t *lbs = p.lb + static_cast<int64_t>(s) * p.nchunk * SCAN_WARPS;
    const BoundMode bm = bound_mode(c, p.chunk, p.m.k_sel);
    const int per = bm.warp_mode ? SCAN_WARPS : 1;  // slots read per chunk
    const int nslot = static_cast<int>(bm.nch) * per;
    uint32_t bound = 0xFFFFFFFFu;
#pragma unroll 4
    for (int i = lane; i < nslot; i += 32)
        bound = min(bound, __ldcg(lbs + (per == 1 ? static_cast<int64_t>(i) * SCAN_WARPS : i)));
    bound = __reduce_min_sync(0xFFFFFFFFu, bound);
    auto keep = [&](int u) {
        return base + u * FILTER_THREADS + threadIdx.x < c && f2key(v[u]) >= bound;
    };
    int mine = 0;
#pragma unroll
    for (int u = 0; u < FILTER_PER_THREAD; ++u) mine += __popc(__ballot_sync(0xFFFFFFFFu, keep(u)));
    if (lane == 0) s_warp[warp] = mine;
    __syncthreads();
    if (threadIdx.x == 0) {
        int tot = 0;
        for (int w = 0; w < FILTER_THREADS / 32; ++w) {
            const int x = s_warp[w];
            s_warp[w] = tot;
            tot += x;
        }
        s_warp[FILTER_THREADS / 32] =
            tot > 0 ? atomicAdd(&p.ccount[static_cast<int64_t>(s) * CCOUNT_STRIDE], tot) : 0;
    }
    __syncthreads();
    int pos = s_warp[FILTER_THREADS / 32] + s_warp[warp];
#pragma unroll
    for (int u = 0; u < FILTER_PER_THREAD; ++u) {
        const int64_t b = base + u * FILTER_THREADS + threadIdx.x;
        const bool k = keep(u);
        const unsigned ball = __ballot_sync(0xFFFFFFFFu, k);
        if (k) {
            const int at = pos + __popc(ball & ltmask);
            if (at < CAND_CAP)
                p.cand[static_cast<int64_t>(s) * CAND_CAP + at] =
                    make_uint2(__float_as_uint(v[u]), static_cast<uint32_t>(b));
            // the decode attention gathers the selected blocks' K and V rows
            // right after the merge; the candidates include them, so their rows
            // are brought into L2 now, while HBM is otherwise idle
            if (p.kpre && at < p.pre_cap) {
                const int64_t off = (static_cast<int64_t>(s) * p.m.max_ctx + b * kBlock) * (kHKV * kD);
                prefetch_l2_bulk(p.kpre + off, kBlock * kHKV * kD * 2);
                prefetch_l2_bulk(p.vpre + off, kBlock * kHKV * kD * 2);
            }
        }
        pos += __popc(ball);
    }
    if (p.kpre && blockIdx.x == 0 && threadIdx.x == 0) {  // the current block is always attended
        const int64_t off = (static_cast<int64_t>(s) * p.m.max_ctx + c * kBlock) * (kHKV * kD);
        prefetch_l2_bulk(p.kpre + off, kBlock * kHKV * kD * 2);
        prefetch_l2_bulk(p.vpre + off, kBlock * kHKV * kD * 2);
    }
}

// One CTA per sequence: the selection row, from the filter's candidates
// (staged in shared memory) or, for rows that need no selection, directly.
__global__ void __launch_bounds__(MERGE_THREADS) merge_kernel(MergeParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint2 *items = reinterpret_cast<uint2 *>(smem);
    uint32_t *sortb = reinterpret_cast<uint32_t *>(items + CAND_CAP);  // [1024]: sort input at 512..
    uint32_t *hist = sortb + 1024;
    int *ctl = reinterpret_cast<int *>(hist + 256);
    pdl_trigger();
    const int s = blockIdx.x;
    // the length (an input of the step) is read while the filter finishes;
    // the row is written only after the wait: before it, the previous step's
    // attention may still be reading the index rows
    const bool trivial = trivial_row<MERGE_THREADS>(p, s, false);
    const int64_t c = (p.seq_lens[s] - 1) / kBlock;
    pdl_wait();  // candidates of the filter (and, through it, the scan's scores)
    if (trivial) {
        trivial_row<MERGE_THREADS>(p, s, true);
        return;
    }
    merge_row<MERGE_THREADS>(p, s, c, items, CAND_CAP, sortb, hist, ctl);
}

}  // namespace dx

DecodePlan decode_plan(int batch, int64_t max_ctx, int sms) {
    DecodePlan pl;
    // Chunks per sequence: batch x chunks should fill the SMs evenly (the
    // scan is bound by HBM bandwidth, so the SM with the most CTAs sets the
    // time), and among even fillings fewer chunks are better: they give a
    // tighter selection bound and so fewer candidates for the merge.
    const int64_t cmax = (max_ctx - 1) / kBlock;
    int64_t nchunk = 1;
    double best = -1.0;
    for (int per_sm = 2; per_sm <= 8; ++per_sm) {
        int64_t n = (static_cast<int64_t>(per_sm) * sms + batch / 2) / batch;
        if (n < 1) n = 1;
        const double ctas = static_cast<double>(batch) * static_cast<double>(n);
        const double eff = ctas / (std::ceil(ctas / sms) * sms);
        if (eff > best + 0.02) {
            best = eff;
            nchunk = n;
        }
    }
    int64_t ch = cmax > 0 ? (cmax + nchunk - 1) / nchunk : 1;
    ch = ((ch + 31) / 32) * 32;
    if (ch < 1024) ch = 1024;
    if (ch > dx::MAX_CHUNK) ch = dx::MAX_CHUNK;
    nchunk = cmax > 0 ? (cmax + ch - 1) / ch : 1;
    if (nchunk > dx::MAX_NCHUNK) {
        ch = (((cmax + dx::MAX_NCHUNK - 1) / dx::MAX_NCHUNK + 31) / 32) * 32;
        nchunk = (cmax + ch - 1) / ch;
    }
    pl.chunk = ch;
    pl.nchunk = static_cast<int>(nchunk < 1 ? 1 : nchunk);
    // attention splits: one wave of CTAs (one per SM: the kernel holds 216 KB
    // of shared memory), as many splits per sequence as fit, at most 16
    int nsplit = sms / batch;
    if (nsplit > 16) nsplit = 16;
    if (nsplit < 1) nsplit = 1;
    pl.nsplit = nsplit;
    return pl;
}

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace of the decode indexer: scores, candidates, counters.
static size_t index_ws_bytes(int batch, int64_t max_ctx) {
    size_t b = 0;
    b += align256(static_cast<size_t>(batch) * (max_ctx / kBlock) * sizeof(float));      // scores
    b += align256(static_cast<size_t>(batch) * dx::CAND_CAP * sizeof(uint2));            // cand
    b += align256(static_cast<size_t>(batch) * dx::CCOUNT_STRIDE * sizeof(int32_t));     // ccount
    b += align256(static_cast<size_t>(batch) * dx::MAX_NCHUNK * (dx::SCAN_THREADS / 32) * sizeof(uint32_t));  // bounds
    return b;
}

size_t decode_ws_bytes(int batch, int64_t max_ctx, int budget, int sms) {
    const DecodePlan pl = decode_plan(batch, max_ctx, sms);
    size_t b = index_ws_bytes(batch, max_ctx);
    b += align256(static_cast<size_t>(batch) * budget * sizeof(int32_t));            // idx
    b += align256(static_cast<size_t>(batch) * pl.nsplit * kHQ * kD * sizeof(float)); // part_o
    b += align256(static_cast<size_t>(batch) * pl.nsplit * kHQ * sizeof(float));      // part_lse
    return b;
}

size_t decode_index_ws_bytes(int batch, int64_t max_ctx) { return index_ws_bytes(batch, max_ctx); }

cudaError_t launch_decode_index(int batch, int64_t max_ctx, const DecodePlan &plan,
                                const uint16_t *qi, const uint16_t *w, const uint16_t *kblk,
                                const int32_t *seq_lens, int budget, void *ws, int32_t *idx_out,
                                int32_t *status, const uint16_t *k_cache, const uint16_t *v_cache,
                                cudaStream_t stream) {
    const int k_sel = budget - 1;
    uint8_t *base = static_cast<uint8_t *>(ws);
    float *scores = reinterpret_cast<float *>(base);
    base += align256(static_cast<size_t>(batch) * (max_ctx / kBlock) * sizeof(float));
    uint2 *cand = reinterpret_cast<uint2 *>(base);
    base += align256(static_cast<size_t>(batch) * dx::CAND_CAP * sizeof(uint2));
    int32_t *ccount = reinterpret_cast<int32_t *>(base);
    base += align256(static_cast<size_t>(batch) * dx::CCOUNT_STRIDE * sizeof(int32_t));
    uint32_t *lb = reinterpret_cast<uint32_t *>(base);
    dx::MergeParams mp;
    mp.seq_lens = seq_lens;
    mp.max_ctx = max_ctx;
    mp.k_sel = k_sel;
    mp.budget = budget;
    mp.scores = scores;
    mp.cand = cand;
    mp.ccount = ccount;
    mp.idx = idx_out;
    mp.status = status;
    cudaError_t e;
    if (k_sel > 0) {
        dx::ScanParams sp;
        sp.qi = qi;
        sp.w = w;
        sp.kblk = kblk;
        sp.seq_lens = seq_lens;
        sp.max_ctx = max_ctx;
        sp.chunk = plan.chunk;
        sp.nchunk = plan.nchunk;
        sp.k_sel = k_sel;
        sp.scores = scores;
        sp.lb = lb;
        sp.ccount = ccount;
        sp.status = status;
        const int smem = static_cast<int>(plan.chunk * 4 + 256 * 4 + 32);
        e = cudaFuncSetAttribute(dx::scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        dx::scan_kernel<<<dim3(plan.nchunk, batch), dx::SCAN_THREADS, smem, stream>>>(sp);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        dx::FilterParams fp;
        fp.m = mp;
        fp.lb = lb;
        fp.nchunk = plan.nchunk;
        fp.chunk = plan.chunk;
        fp.cand = cand;
        fp.ccount = ccount;
        // prefetch while the candidates' K and V rows fit in L2 beside the
        // scores: about twice the budget per sequence, 8 KiB per block
        const bool pre = static_cast<int64_t>(batch) * 2 * budget * 2 * kBlock * kHKV * kD * 2 <= dx::kPrefetchL2Bytes;
        fp.kpre = pre ? k_cache : nullptr;
        fp.vpre = pre ? v_cache : nullptr;
        fp.pre_cap = 2 * budget;
        const int64_t cmax = (max_ctx - 1) / kBlock;
        const int64_t per_cta = static_cast<int64_t>(dx::FILTER_THREADS) * dx::FILTER_PER_THREAD;
        const int64_t fx = cmax > 0 ? (cmax + per_cta - 1) / per_cta : 1;
        e = launch_pdl(dx::filter_kernel, dim3(static_cast<unsigned>(fx), batch), dim3(dx::FILTER_THREADS), 0,
                       stream, fp);
        if (e != cudaSuccess) return e;
    }
    const int smem = dx::CAND_CAP * 8 + 1024 * 4 + 256 * 4 + 8 * 4;
    e = cudaFuncSetAttribute(dx::merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(dx::merge_kernel, dim3(batch), dim3(dx::MERGE_THREADS), static_cast<size_t>(smem), stream,
                      mp);
}

}  // namespace qsa
