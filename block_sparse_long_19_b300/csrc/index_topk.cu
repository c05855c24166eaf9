// Prefill indexer with fused selection, on the 5th-generation tensor cores.
//
// What it computes (Qwen3.8-Flash-Next launch post, "Model Architecture /
// Attention: GDN + QSA"; shapes from the model card, "Model Overview / Qwen
// Sparse Attention"): for every query t and every complete past block
// b < c(t) = floor(t/4),
//     s[t,b] = sum_{h<4} w[t,h] * max(0, qi[t,h] . kblk[b]),
// and the selection keeps block c(t) plus the (budget-1) past blocks with
// the highest s (ties: lower block first).  The score matrix is never
// written to memory.
//
// Design (one persistent CTA per SM, 20 warps):
//   * the contraction runs "swap-AB": the MMA's M = 128 block keys (A, from a
//     TMA tile of kblk), N = 256 columns = 64 query tokens x 4 indexer heads
//     (B, a TMA tile of qi that stays resident for the whole query tile),
//     K = 128; fp32 accumulators live in TMEM, double-buffered (2 x 256 cols);
//   * warp 0 issues the TMA loads, warp 1 issues tcgen05.mma (one thread),
//     warp 2 owns the TMEM allocation, warps 4..19 are the epilogue: four
//     groups of four warps, group g owning tokens 16g .. 16g+15 and warp q of
//     a group TMEM lane quarter q (32 blocks of the tile).  A thread reads the
//     4 head columns of each of its 16 tokens, forms the score and tests it
//     against the token's running threshold;
//   * selection is an exact streaming top-k: every token keeps a candidate
//     list (global workspace, mostly L2-resident) of the blocks that beat its
//     threshold.  Every second tile a group checks its lists; one that could
//     overflow is cut back by the group's 128 threads together: a radix
//     select finds a bound at or below the k-th best (score desc, index asc),
//     the survivors are written back and the threshold is raised to it.
//     Block tiles are visited in ascending block order, so a later block with
//     a score equal to the threshold always loses the tie and is never needed;
//   * after the last block tile the group selects each token's final k
//     exactly, sorts them by block index (bitonic, in registers) and writes
//     the row.
#include <type_traits>

#include "qsa_common.cuh"
#include "qsa_kernels.h"
#include "qsa_select.cuh"

namespace qsa {
namespace ix {

constexpr int TQ = 64;               // query tokens per tile
constexpr int NCOL = TQ * kHI;       // 256 MMA columns (token-major, head-minor)
constexpr int TB = 128;              // block keys per block tile (MMA M)
constexpr int NSTAGE = 3;            // kblk tile ring
constexpr int CAP = 2048;            // candidate slots per token
constexpr int SUB = CAP / 4;         // per-warp sub-list of a token (one per TMEM lane quarter)
constexpr int KSTEPS = kDI / 16;     // 8 MMAs of K = 16
constexpr int NGRP = 4;              // epilogue groups
constexpr int GTOK = TQ / NGRP;      // 16 tokens (64 TMEM columns) per group
constexpr int NEPI = 4 * NGRP;       // 16 epilogue warps: group x TMEM lane quarter
constexpr int GT = 128;              // threads per group
constexpr int THREADS = (4 + NEPI) * 32;
#ifndef QSA_IX_CHK
#define QSA_IX_CHK 2
#endif
#ifndef QSA_IX_FIRST_AT
#define QSA_IX_FIRST_AT 160
#endif
#ifndef QSA_IX_R_MIN
#define QSA_IX_R_MIN 64
#endif
#ifndef QSA_IX_MARGIN
#define QSA_IX_MARGIN 2
#endif
constexpr int CHK = QSA_IX_CHK;      // tiles between list checks
constexpr int FLAG_AT = SUB - 32 * CHK;  // a sub-list longer than this is cut back at a check
constexpr int FIRST_AT = QSA_IX_FIRST_AT;  // before the first prediction: cut back a sub-list beyond this
constexpr int R_MIN = QSA_IX_R_MIN;        // smallest rank a threshold is predicted from
constexpr int MARGIN = QSA_IX_MARGIN;      // predicted thresholds keep MARGIN x (budget-1) blocks
constexpr int HIST_INTS = 4 * 256;   // per group: 3 rotating histogram slots + one for a second rank
constexpr int CTL_INTS = 3 * 16;     // per group: 3 rotating control slots

constexpr int GCOL = GTOK * kHI;     // 64 MMA columns per group
constexpr uint32_t IDESC = idesc_bf16_f32(TB, NCOL);

constexpr int SQ_BYTES = 2 * NCOL * 128;     // two 64-wide K halves, 128-B rows
constexpr int SK_BYTES = 2 * TB * 128;
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + SQ_BYTES;
constexpr int OFF_HIST = OFF_K + NSTAGE * SK_BYTES;
constexpr int OFF_CTL = OFF_HIST + NGRP * HIST_INTS * 4;
constexpr int OFF_SORT = OFF_CTL + NGRP * CTL_INTS * 4;  // per group: 1024 sort slots of 8 bytes
constexpr int OFF_W = OFF_SORT + NGRP * 1024 * 8;
constexpr int OFF_THETA = OFF_W + TQ * 4 * 4;
constexpr int OFF_CNT = OFF_THETA + TQ * 4;      // [4 quarters][TQ] sub-list counts
constexpr int OFF_FLAG = OFF_CNT + 4 * TQ * 4;   // [NGRP groups][2 parities] token masks
constexpr int OFF_PRED = OFF_FLAG + NGRP * 2 * 4;  // [TQ] predicted threshold per token (-inf: none)
constexpr int OFF_GPRED = OFF_PRED + TQ * 4;     // [NGRP] this tile's prediction switch per group
constexpr int OFF_BAR = OFF_GPRED + NGRP * 4;
constexpr int NBAR = 2 * NSTAGE + 2 + 4;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");

struct Params {
    int64_t L;          // end position: queries are tokens q_off .. L-1
    int64_t unit_rows;  // rows of the unit-key tensor map (debug checks)
    int64_t q_off;      // position of the first query row (a cached prefix before it)
    int bshift;         // log2 of the tokens per selection unit: 2 (4-token blocks) or 0 (tokens)
    int nq;
    int k_sel;          // budget - 1
    int budget;
    const uint16_t *w;  // [L - q_off, 4]
    int32_t *idx;       // [L - q_off, budget]
    float *score;       // [L - q_off, budget] or null
    float *dense;       // [L, L/4] (dense mode)
    int64_t dense_ld;
    uint2 *cand;        // [grid, TQ, CAP] {score bits, block}
    int32_t *status;
    int predict;        // raise thresholds by prediction (with the exactness check below)
    uint8_t *redo;      // [nq, 4 groups] set where a prediction failed its check (or null)
    int redo_pass;      // 1: process only the query tiles flagged in redo, without prediction
    int *stop;          // set once a prediction failed anywhere in the call: no more predictions
};

// In the pass after a predicting launch only the flagged query tiles run.
__device__ __forceinline__ bool tile_skipped(const Params &p, int q) {
    return p.redo_pass && *reinterpret_cast<const uint32_t *>(p.redo + 4 * static_cast<int64_t>(q)) == 0u;
}

// A TMEM load of 16 columns (32 lanes x 32 bit), and the wait for every
// outstanding TMEM load.  The chunk loop issues chunk ch+1's load before
// chunk ch's arithmetic and waits after it, so the load's latency is hidden.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
// The wait names r (the registers of the load in flight) as in-out operands,
// so no use of them can move above it.
__device__ __forceinline__ void tmem_wait16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
                   "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// Bounded wait on an mbarrier phase that gives the issue slots away while it
// waits: after a failed test the warp sleeps (nanosleep takes it off the
// scheduler), so a waiting warp does not compete with the warps that score.
// The clock is read only every 64 tries.
template <int SLEEP_NS>
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity) {
    auto try_once = [&]() {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        return done != 0;
    };
    if (try_once()) return true;
    const unsigned long long t0 = globaltimer();
    for (unsigned n = 1;; ++n) {
        __nanosleep(SLEEP_NS);
        if (try_once()) return true;
        if ((n & 63u) == 0 && globaltimer() - t0 > kWaitLimitNs) return false;
    }
}

// Barrier among the 4 warps (128 threads) of one epilogue group that is also a
// vote: every thread gets the OR of all `fail` flags, so a group always
// leaves together (a warp that left alone would strand the others at the next
// barrier; every wait before a barrier is bounded).
__device__ __forceinline__ bool group_sync_fail(int id, bool fail) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, 128, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(fail ? 1 : 0), "r"(id)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void group_bar(int id) {
    asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}

// Block tiles query tile q has to visit: blocks 0 .. c(t_last)-1.
__device__ __forceinline__ int num_btiles(const Params &p, int q) {
    int64_t t_last = p.q_off + static_cast<int64_t>(q) * TQ + TQ - 1;
    if (t_last > p.L - 1) t_last = p.L - 1;
    const int64_t cmax = t_last >> p.bshift;  // units 0..cmax-1 are scored
    return static_cast<int>((cmax + TB - 1) / TB);
}

// A token's candidate list is 4 sub-lists of SUB entries, one per epilogue
// warp of its group (the warp that owns TMEM lane quarter q appends to
// sub-list q with a warp-private count, so appending needs neither atomics
// nor shuffles).  Entries are (score bits, block).  Selection work on a list
// is done by the group's 128 threads together, each warp holding its own
// sub-list in registers (lane l: entries l + 32 i, i < IPL) with the score
// bits turned into order keys.
constexpr int IPL = SUB / 32;  // list entries per lane
constexpr int KEEP_MAX = 768;  // a lower-bound compaction must keep at most this many
static_assert(FLAG_AT + 32 * CHK <= SUB, "a sub-list takes at most 32 entries per tile");
static_assert((KEEP_MAX + 3) / 4 < FLAG_AT, "a compacted list must leave room");

struct StagedRule {
    uint32_t thr_key;
    uint32_t thr_nblk;
    int by_bucket;  // 1: keep key >= thr_key
};

__device__ __forceinline__ bool staged_keep(const StagedRule &r, uint2 it) {
    if (r.by_bucket) return it.x >= r.thr_key;
    return it.x > r.thr_key || (it.x == r.thr_key && ~it.y >= r.thr_nblk);
}

// The group's cooperative steps.  Every step ends in one barrier of the
// group's 128 threads; step s keeps its data in slot s % 3 (a 256-counter
// histogram and 16 control ints) and, before its barrier, clears the
// histogram of slot (s + 1) % 3 for the step after it.  That slot was last
// read in step s - 2, which every thread finished before the barrier of step
// s - 1, so one barrier per step suffices.  `step` counts in every thread
// alike.
struct Group {
    uint32_t *hist;  // [3][256]
    int *ctl;        // [3][16]
    int tg, lane, gw, bar;
    uint32_t step;
};

__device__ __forceinline__ int group_step_begin(Group &G) {
    const int s = static_cast<int>(G.step % 3u);
    uint32_t *nh = G.hist + ((G.step + 1u) % 3u) * 256;
    nh[G.tg] = 0u;
    nh[G.tg + GT] = 0u;
    return s;
}
__device__ __forceinline__ void group_step_end(Group &G) {
    group_bar(G.bar);
    ++G.step;
}

// Loads this warp's sub-list (n entries) into registers as (key, block).
__device__ __forceinline__ void group_load(const uint2 *__restrict__ lst, int n, uint2 (&it)[IPL], int lane) {
#pragma unroll
    for (int i = 0; i < IPL; ++i) {
        const bool v = lane + 32 * i < n;
        it[i] = v ? __ldcg(lst + lane + 32 * i) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < IPL; ++i) it[i].x = f2key(__uint_as_float(it[i].x));
}

// Group radix over the register-held items (contract of warp_radix in
// qsa_select.cuh).  NEG ranks ~block instead of the key; TIE restricts the
// items to those whose key equals tie_key.  n: this warp's item count.
template <bool NEG, bool TIE>
__device__ __forceinline__ RadixOut group_radix(const uint2 (&it)[IPL], int n, uint32_t tie_key, int k,
                                                int max_passes, Group &G) {
    auto item = [&](int i, uint32_t &v) {
        v = NEG ? ~it[i].y : it[i].x;
        return G.lane + 32 * i < n && (!TIE || it[i].x == tie_key);
    };
    uint32_t mx = 0u, mn = 0xFFFFFFFFu;
    int nv = 0;
#pragma unroll
    for (int i = 0; i < IPL; ++i) {
        if (32 * i >= n) break;
        uint32_t v;
        if (item(i, v)) {
            mx = max(mx, v);
            mn = min(mn, v);
            ++nv;
        }
    }
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    mn = __reduce_min_sync(0xFFFFFFFFu, mn);
    nv = __reduce_add_sync(0xFFFFFFFFu, nv);
    {
        const int s = group_step_begin(G);
        int *c = G.ctl + s * 16;
        if (G.lane == 0) {
            c[8 + G.gw] = static_cast<int>(mx);
            c[12 + G.gw] = static_cast<int>(mn);
            c[4 + G.gw] = nv;
        }
        group_step_end(G);
        mx = 0u;
        mn = 0xFFFFFFFFu;
        nv = 0;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            mx = max(mx, static_cast<uint32_t>(c[8 + w]));
            mn = min(mn, static_cast<uint32_t>(c[12 + w]));
            nv += c[4 + w];
        }
    }
    RadixOut r;
    r.krem = k;
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
        const unsigned long long want = prefix >> (lo + w);
        const int s = group_step_begin(G);
        uint32_t *h = G.hist + s * 256;
#pragma unroll
        for (int i = 0; i < IPL; ++i) {
            if (32 * i >= n) break;
            uint32_t v;
            if (item(i, v) && (static_cast<unsigned long long>(v) >> (lo + w)) == want)
                atomicAdd(&h[(v >> lo) & dmask], 1u);
        }
        group_step_end(G);
        // every warp finds the digit itself (no second barrier)
        uint32_t cnt[8];
        uint32_t sum = 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            cnt[b] = h[255 - (G.lane * 8 + b)];
            sum += cnt[b];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (G.lane >= o) incl += t;
        }
        const uint32_t excl = incl - sum;
        const bool mine = excl < static_cast<uint32_t>(r.krem) && static_cast<uint32_t>(r.krem) <= incl;
        int digit = 0;
        uint32_t above = 0, e = 0;
        if (mine) {
            uint32_t acc = excl;
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                if (acc + cnt[b] >= static_cast<uint32_t>(r.krem)) {
                    digit = 255 - (G.lane * 8 + b);
                    above = acc;
                    e = cnt[b];
                    break;
                }
                acc += cnt[b];
            }
        }
        const int src = __ffs(__ballot_sync(0xFFFFFFFFu, mine)) - 1;
        digit = __shfl_sync(0xFFFFFFFFu, digit, src);
        above = __shfl_sync(0xFFFFFFFFu, above, src);
        e = __shfl_sync(0xFFFFFFFFu, e, src);
        r.krem -= static_cast<int>(above);
        eq = static_cast<int>(e);
        prefix |= static_cast<unsigned long long>(digit) << lo;
        if (eq == r.krem) break;
    }
    r.thr = static_cast<uint32_t>(prefix);
    r.eq = eq;
    r.lo = lo;
    return r;
}

// Digit search of one radix pass (every warp does it itself from the
// finished histogram h, no barrier): the bucket of the k-th largest value.
__device__ __forceinline__ void radix_digit(const uint32_t *h, int lane, int krem, int &digit, uint32_t &above,
                                            uint32_t &e) {
    uint32_t cnt[8];
    uint32_t sum = 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        cnt[b] = h[255 - (lane * 8 + b)];
        sum += cnt[b];
    }
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
    }
    const uint32_t excl = incl - sum;
    const bool mine = excl < static_cast<uint32_t>(krem) && static_cast<uint32_t>(krem) <= incl;
    digit = 0;
    above = 0;
    e = 0;
    if (mine) {
        uint32_t acc = excl;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            if (acc + cnt[b] >= static_cast<uint32_t>(krem)) {
                digit = 255 - (lane * 8 + b);
                above = acc;
                e = cnt[b];
                break;
            }
            acc += cnt[b];
        }
    }
    const int src = __ffs(__ballot_sync(0xFFFFFFFFu, mine)) - 1;
    digit = __shfl_sync(0xFFFFFFFFu, digit, src);
    above = __shfl_sync(0xFFFFFFFFu, above, src);
    e = __shfl_sync(0xFFFFFFFFu, e, src);
}

// group_radix<false, false>(it, n, 0, k, 2, G) for two ranks k1 and k2 at
// once (the same two results): the max / min step and the first pass are
// shared, and the second pass counts both ranks' buckets in one step, so the
// pair takes 3 group steps instead of 6.
__device__ __forceinline__ void group_radix2(const uint2 (&it)[IPL], int n, int k1, int k2, Group &G, RadixOut &r1,
                                             RadixOut &r2) {
    uint32_t mx = 0u, mn = 0xFFFFFFFFu;
    int nv = 0;
#pragma unroll
    for (int i = 0; i < IPL; ++i) {
        if (32 * i >= n) break;
        if (G.lane + 32 * i < n) {
            mx = max(mx, it[i].x);
            mn = min(mn, it[i].x);
            ++nv;
        }
    }
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    mn = __reduce_min_sync(0xFFFFFFFFu, mn);
    nv = __reduce_add_sync(0xFFFFFFFFu, nv);
    {
        const int s = group_step_begin(G);
        int *c = G.ctl + s * 16;
        if (G.lane == 0) {
            c[8 + G.gw] = static_cast<int>(mx);
            c[12 + G.gw] = static_cast<int>(mn);
            c[4 + G.gw] = nv;
        }
        group_step_end(G);
        mx = 0u;
        mn = 0xFFFFFFFFu;
        nv = 0;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            mx = max(mx, static_cast<uint32_t>(c[8 + w]));
            mn = min(mn, static_cast<uint32_t>(c[12 + w]));
            nv += c[4 + w];
        }
    }
    r1.krem = k1;
    r2.krem = k2;
    if (mx == mn) {
        r1.thr = r2.thr = mx;
        r1.eq = r2.eq = nv;
        r1.lo = r2.lo = 0;
        return;
    }
    const int hi = 32 - __clz(mx ^ mn);
    const unsigned long long prefix0 = hi >= 32 ? 0ull : (static_cast<unsigned long long>(mx >> hi) << hi);
    unsigned long long pre1 = prefix0, pre2 = prefix0;
    int lo = hi;
    int eq1 = nv, eq2 = nv;
    bool go1 = true, go2 = true;  // the rank still refines its bucket
    uint32_t *aux = G.hist + 3 * 256;
    for (int pass = 0; pass < 2 && lo > 0 && (go1 || go2); ++pass) {
        const int w = lo >= 8 ? 8 : lo;
        lo -= w;
        const uint32_t dmask = (1u << w) - 1u;
        const unsigned long long want1 = pre1 >> (lo + w), want2 = pre2 >> (lo + w);
        const bool split = go1 && go2 && want1 != want2;  // two buckets to count
        const int s = group_step_begin(G);
        if (pass == 0) {  // the second pass's extra histogram starts from zero
            aux[G.tg] = 0u;
            aux[G.tg + GT] = 0u;
        }
        uint32_t *h = G.hist + s * 256;
        uint32_t *h2 = split ? aux : h;
        const unsigned long long wa = go1 ? want1 : want2;
#pragma unroll
        for (int i = 0; i < IPL; ++i) {
            if (32 * i >= n) break;
            const uint32_t v = it[i].x;
            if (G.lane + 32 * i < n) {
                const unsigned long long top = static_cast<unsigned long long>(v) >> (lo + w);
                if (top == wa) atomicAdd(&h[(v >> lo) & dmask], 1u);
                else if (split && top == want2) atomicAdd(&h2[(v >> lo) & dmask], 1u);
            }
        }
        group_step_end(G);
        if (go1) {
            int digit;
            uint32_t above, e;
            radix_digit(h, G.lane, r1.krem, digit, above, e);
            r1.krem -= static_cast<int>(above);
            eq1 = static_cast<int>(e);
            pre1 |= static_cast<unsigned long long>(digit) << lo;
            r1.lo = lo;
            if (eq1 == r1.krem) go1 = false;
        }
        if (go2) {
            int digit;
            uint32_t above, e;
            radix_digit(split ? aux : h, G.lane, r2.krem, digit, above, e);
            r2.krem -= static_cast<int>(above);
            eq2 = static_cast<int>(e);
            pre2 |= static_cast<unsigned long long>(digit) << lo;
            r2.lo = lo;
            if (eq2 == r2.krem) go2 = false;
        }
    }
    r1.thr = static_cast<uint32_t>(pre1);
    r1.eq = eq1;
    r2.thr = static_cast<uint32_t>(pre2);
    r2.eq = eq2;
}

// Exact k best (key desc, block asc) of the group's items, plus the
// streaming threshold a later (higher-index) block must reach: s >= *theta.
__device__ __forceinline__ StagedRule group_select_exact(const uint2 (&it)[IPL], int n, int k, Group &G,
                                                         float *theta) {
    const RadixOut r = group_radix<false, false>(it, n, 0u, k, 8, G);
    StagedRule rule;
    rule.thr_key = r.thr;
    rule.thr_nblk = 0;
    rule.by_bucket = 1;
    if (r.eq == r.krem) {
        *theta = r.lo == 0 ? nextafterf(key2f(r.thr), INFINITY) : key2f(r.thr);
        return rule;
    }
    // the k-th key is exactly r.thr; take the r.krem ties with the lowest blocks
    const RadixOut r2 = group_radix<true, true>(it, n, r.thr, r.krem, 8, G);
    rule.by_bucket = 0;
    rule.thr_nblk = r2.thr;
    *theta = nextafterf(key2f(r.thr), INFINITY);
    return rule;
}

// Hands every kept item to emit(item, rank), ranks counted warp by warp
// (then entry order within the warp); returns the number kept.  One step.
template <typename Keep, typename Emit>
__device__ __forceinline__ int group_ranks_apply(const uint2 (&it)[IPL], int n, Keep keep, Emit emit, Group &G) {
    int mine = 0;
#pragma unroll
    for (int i = 0; i < IPL; ++i) {
        if (32 * i >= n) break;
        mine += __popc(__ballot_sync(0xFFFFFFFFu, G.lane + 32 * i < n && keep(it[i])));
    }
    const int s = group_step_begin(G);
    int *c = G.ctl + s * 16;
    if (G.lane == 0) c[G.gw] = mine;
    group_step_end(G);
    const int4 cw = *reinterpret_cast<const int4 *>(c);
    int run = (G.gw > 0 ? cw.x : 0) + (G.gw > 1 ? cw.y : 0) + (G.gw > 2 ? cw.z : 0);
    const unsigned ltmask = (1u << G.lane) - 1u;
#pragma unroll
    for (int i = 0; i < IPL; ++i) {
        if (32 * i >= n) break;
        const bool kp = G.lane + 32 * i < n && keep(it[i]);
        const unsigned ball = __ballot_sync(0xFFFFFFFFu, kp);
        if (kp) emit(it[i], run + __popc(ball & ltmask));
        run += __popc(ball);
    }
    return cw.x + cw.y + cw.z + cw.w;
}

// Number of the group's items for which keep(item) holds.  One step.
template <typename Keep>
__device__ __forceinline__ int group_count(const uint2 (&it)[IPL], int n, Keep keep, Group &G) {
    int mine = 0;
#pragma unroll
    for (int i = 0; i < IPL; ++i) {
        if (32 * i >= n) break;
        mine += __popc(__ballot_sync(0xFFFFFFFFu, G.lane + 32 * i < n && keep(it[i])));
    }
    const int s = group_step_begin(G);
    int *c = G.ctl + s * 16;
    if (G.lane == 0) c[G.gw] = mine;
    group_step_end(G);
    const int4 cw = *reinterpret_cast<const int4 *>(c);
    return cw.x + cw.y + cw.z + cw.w;
}

// Store only where pred holds, as a predicated instruction (no branch).  No
// "memory" clobber: the compiler may move other loads across it (ordering
// against the list readers comes from the group barrier).
__device__ __forceinline__ void st_global_pred(uint2 *addr, uint2 v, bool pred) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t@p st.global.v2.b32 [%1], {%2, %3};\n\t}" ::"r"(
            pred ? 1 : 0),
        "l"(addr), "r"(v.x), "r"(v.y));
}

template <bool DENSE>
__global__ void __launch_bounds__(THREADS, 1)
    index_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                 Params p) {
    extern __shared__ uint8_t smem_raw[];
    // aligned by pointer arithmetic on the shared array itself (a round trip
    // through an integer would hide the state space and turn every access
    // into a generic one)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sQ = smem + OFF_Q;
    uint8_t *sK = smem + OFF_K;
    int *sCtl = reinterpret_cast<int *>(smem + OFF_CTL);
    uint32_t *sHist = reinterpret_cast<uint32_t *>(smem + OFF_HIST);
    unsigned long long *sSort = reinterpret_cast<unsigned long long *>(smem + OFF_SORT);
    float *sW = reinterpret_cast<float *>(smem + OFF_W);
    float *sTheta = reinterpret_cast<float *>(smem + OFF_THETA);
    float *sPred = reinterpret_cast<float *>(smem + OFF_PRED);
    volatile int *sGPred = reinterpret_cast<volatile int *>(smem + OFF_GPRED);
    int *sCnt = reinterpret_cast<int *>(smem + OFF_CNT);  // sCnt[q * TQ + tl]
    unsigned *sFlag = reinterpret_cast<unsigned *>(smem + OFF_FLAG);  // sFlag[group * 2 + parity]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint64_t *full = bars;
    uint64_t *empty = bars + NSTAGE;
    uint64_t *qfull = bars + 2 * NSTAGE;
    uint64_t *qempty = qfull + 1;
    uint64_t *tfull = qfull + 2;   // [2]
    uint64_t *tempty = qfull + 4;  // [2]
    volatile uint32_t *sMisc = reinterpret_cast<volatile uint32_t *>(smem + OFF_MISC);
    // sMisc[0] = TMEM base, sMisc[1] = abort flag

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(qfull, 1);
        mbar_init(qempty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], NEPI);
        }
        sMisc[1] = 0;
        sMisc[2] = 0;  // set once a group's prediction failed: the CTA stops predicting
        for (int i = 0; i < NGRP * 2; ++i) sFlag[i] = 0u;
        fence_barrier_init();
    }
    if (warp == 2) {
        tmem_alloc(const_cast<uint32_t *>(&sMisc[0]), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = sMisc[0];

    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            uint32_t st = 0, ph = 0, qph = 0;
            bool ok = true;
            for (int kk = blockIdx.x; kk < p.nq && ok; kk += gridDim.x) {
                const int q = p.nq - 1 - kk;
                const int nbt = num_btiles(p, q);
                if (nbt == 0 || tile_skipped(p, q)) continue;
                if (!mbar_wait(qempty, qph ^ 1)) { ok = false; break; }
                qph ^= 1;
                mbar_arrive_expect_tx(qfull, SQ_BYTES);
                tma_load_2d(sQ, &map_q, qfull, 0, q * NCOL);
                tma_load_2d(sQ + SQ_BYTES / 2, &map_q, qfull, 64, q * NCOL);
                for (int j = 0; j < nbt; ++j) {
                    if (sMisc[1]) { ok = false; break; }
                    if (!mbar_wait_sleep<256>(&empty[st], ph ^ 1)) { ok = false; break; }
                    uint8_t *dst = sK + st * SK_BYTES;
                    debug_check(p.status, static_cast<int64_t>(j) * TB < p.unit_rows);  // tile starts inside the map
                    mbar_arrive_expect_tx(&full[st], SK_BYTES);
                    tma_load_2d(dst, &map_k, &full[st], 0, j * TB);
                    tma_load_2d(dst + SK_BYTES / 2, &map_k, &full[st], 64, j * TB);
                    if (++st == NSTAGE) { st = 0; ph ^= 1; }
                }
            }
            if (!ok) {
                report(p.status, QSA_ERR_TIMEOUT);
                sMisc[1] = 1;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer --
        if (lane == 0) {
            uint32_t st = 0, ph = 0, qph = 0, acc = 0, qcommits = 0;
            bool ok = true;
            const uint32_t sq_addr = smem_u32(sQ);
            const uint32_t sk_addr = smem_u32(sK);
            for (int kk = blockIdx.x; kk < p.nq && ok; kk += gridDim.x) {
                const int q = p.nq - 1 - kk;
                const int nbt = num_btiles(p, q);
                if (nbt == 0 || tile_skipped(p, q)) continue;
                if (!mbar_wait(qfull, qph)) { ok = false; break; }
                qph ^= 1;
                tc_fence_after();
                for (int j = 0; j < nbt; ++j) {
                    if (sMisc[1]) { ok = false; break; }
                    const uint32_t buf = acc & 1;
                    const uint32_t use = acc >> 1;
                    if (!mbar_wait_sleep<64>(&tempty[buf], (use & 1) ^ 1)) { ok = false; break; }
                    if (!mbar_wait_sleep<64>(&full[st], ph)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d = tmem_base + buf * NCOL;
#pragma unroll
                    for (int kx = 0; kx < KSTEPS; ++kx) {
                        const uint32_t half = kx >> 2, off = (kx & 3) * 32;
                        const uint64_t ad = sdesc_sw128(sk_addr + st * SK_BYTES + half * (SK_BYTES / 2) + off);
                        const uint64_t bd = sdesc_sw128(sq_addr + half * (SQ_BYTES / 2) + off);
                        tc_mma_bf16(d, ad, bd, IDESC, kx > 0 ? 1u : 0u);
                    }
                    tc_commit(&empty[st]);
                    tc_commit(&tfull[buf]);
                    if (++st == NSTAGE) { st = 0; ph ^= 1; }
                    ++acc;
                }
                tc_commit(qempty);
                ++qcommits;
            }
            // the CTA must not exit before its last commit has arrived
            if (ok && qcommits > 0 && !mbar_wait(qempty, (qcommits - 1) & 1)) ok = false;
            if (!ok) {
                report(p.status, QSA_ERR_TIMEOUT);
                sMisc[1] = 1;
            }
        }
    } else if (warp >= 4) {
        // --------------------------------------------------- epilogue --
        // 16 warps = 4 groups x 4 TMEM lane quarters; group g scores tokens
        // g*16 .. g*16+15 (TMEM columns g*64 .. g*64+63) for the 128 blocks of
        // a tile; the group's 128 threads together do its selection work.
        const int e = warp - 4;
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        const int g = e >> 2;          // group
        const int tg = quarter * 32 + lane;  // thread index within the group
        const int bar = 1 + g;         // hardware barrier id of the group
        Group G{sHist + g * HIST_INTS, sCtl + g * CTL_INTS, tg, lane, quarter, 1 + g, 0u};
        unsigned long long *sort64 = sSort + g * 1024;  // [0..511] exchange, [512..1023] input
        uint32_t *sort32 = reinterpret_cast<uint32_t *>(sort64);
        const unsigned ltmask = (1u << lane) - 1u;
        // this warp's sub-lists: token tl's at sub[tl * CAP]
        uint2 *sub = p.cand + static_cast<int64_t>(blockIdx.x) * TQ * CAP + quarter * SUB;
        uint32_t acc = 0, nchk = 0;
        bool ok = true;
        // thresholds are predicted until a prediction fails its check anywhere
        // in the CTA or the call: rows whose scores are not spread alike over
        // their blocks (a structured context) then run the plain streaming
        // selection, and few query tiles are redone.  The switch is read once
        // per tile for the whole group (group-uniform).
        bool predict_on = p.predict != 0;
        for (int kk = blockIdx.x; kk < p.nq; kk += gridDim.x) {
            const int q = p.nq - 1 - kk;
            // positions fit in 32 bits (at most 2^24 tokens): the epilogue runs
            // at its register limit, and 64-bit copies cost it scheduling room
            const int t0 = static_cast<int>(p.q_off) + q * TQ;
            const int L32 = static_cast<int>(p.L);
            const int nbt = num_btiles(p, q);
            if (tile_skipped(p, q)) continue;
            if (group_sync_fail(bar, !ok || sMisc[1] != 0)) { ok = false; break; }
            if (tg < GTOK) {
                const int tl = g * GTOK + tg;
                const int t = t0 + tl;
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) sCnt[qq * TQ + tl] = 0;
                sTheta[tl] = -INFINITY;
                sPred[tl] = -INFINITY;
                if (tg == 0)
                    sGPred[g] = predict_on && sMisc[2] == 0u &&
                                (p.stop == nullptr || *reinterpret_cast<volatile int *>(p.stop) == 0);
#pragma unroll
                for (int h = 0; h < kHI; ++h) {
                    float wv = 0.f;
                    if (t < L32) wv = __uint_as_float(static_cast<uint32_t>(p.w[static_cast<int64_t>(t - static_cast<int>(p.q_off)) * kHI + h]) << 16);
                    // w / 2 (exact for every bf16 w), see the score below
                    sW[(tl >> 2) * 16 + h * 4 + (tl & 3)] = 0.5f * wv;  // [token quad][head][token]
                }
            }
            if (group_sync_fail(bar, false)) { ok = false; break; }
            predict_on = sGPred[g] != 0;
            const bool tile_all_in = (t0 + TQ <= L32);
            const int c_min = t0 >> p.bshift;
            for (int j = 0; j < nbt; ++j) {
                const uint32_t buf = acc & 1;
                const uint32_t use = acc >> 1;
                // lists are checked every CHK tiles and after the last one (that
                // vote also makes sure the whole group goes on to the selection)
                const bool last = j == nbt - 1;
                const bool check = !DENSE && (last || (j + 1) % CHK == 0);
                if (ok && !mbar_wait_sleep<64>(&tfull[buf], use & 1)) ok = false;
                if (!ok) {  // skip the work, keep taking part in the votes
                    ++acc;
                    if (check && group_sync_fail(bar, true)) break;
                    continue;
                }
                tc_fence_after();
                const int b = j * TB + quarter * 32 + lane;
                const bool masked = !(tile_all_in && (j * TB + TB <= c_min));
                const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       buf * NCOL + static_cast<uint32_t>(g * GCOL);
                // 4 chunks of 4 tokens (16 columns each), each chunk's TMEM load
                // in flight during the arithmetic of the chunk before it
                uint32_t curb[2][16];
                // MASKED: the tile holds blocks that some of the tokens may not see
                auto score_tile = [&](auto masked_c) {
                    constexpr bool MASKED = decltype(masked_c)::value;
                    tmem_ld16(tbase, curb[0]);
                    tmem_wait16(curb[0]);
#pragma unroll
                    for (int ch = 0; ch < GTOK / 4; ++ch) {
                        uint32_t (&cur)[16] = curb[ch & 1];
                        if (ch + 1 < GTOK / 4) tmem_ld16(tbase + (ch + 1) * 16, curb[(ch + 1) & 1]);
                        const int tl0 = g * GTOK + ch * 4;
                        // s = sum_h w_h * max(0, x_h) for two tokens per packed FMA,
                        // heads in order 0..3, the first product added to +0 (the
                        // sum is never -0); per component this is plain fmaf.
                        // max(0, x) is taken as x + |x| = 2 max(0, x) (exact: a
                        // doubling or x - x = +0), the 2 cancelled by the halved
                        // weight, so the product w/2 * (x + |x|) is exactly
                        // w * max(0, x) and each fmaf rounds as before; the add
                        // runs on the FMA pipe, where a max would take the
                        // integer pipe that the threshold tests and list pushes
                        // also need.  (Exact for |x| < 2^127; a dot product of
                        // bf16 vectors beyond that is out of range anyway.)
                        float2 s01 = make_float2(0.f, 0.f), s23 = make_float2(0.f, 0.f);
#pragma unroll
                        for (int h = 0; h < kHI; ++h) {
                            const float4 wv = *reinterpret_cast<const float4 *>(&sW[(tl0 >> 2) * 16 + h * 4]);
                            auto two_relu = [](uint32_t u) {
                                const float x = __uint_as_float(u);
                                return __fadd_rn(x, fabsf(x));
                            };
                            const float2 x01 = make_float2(two_relu(cur[h]), two_relu(cur[4 + h]));
                            const float2 x23 = make_float2(two_relu(cur[8 + h]), two_relu(cur[12 + h]));
                            s01 = __ffma2_rn(make_float2(wv.x, wv.y), x01, s01);
                            s23 = __ffma2_rn(make_float2(wv.z, wv.w), x23, s23);
                        }
                        const float sv[4] = {s01.x, s01.y, s23.x, s23.y};
                        if constexpr (DENSE) {
#pragma unroll
                            for (int tk = 0; tk < 4; ++tk) {
                                const int t = t0 + tl0 + tk;
                                const bool valid = !MASKED || ((t < L32) && (b < (t >> p.bshift)));
                                if (valid) p.dense[static_cast<int64_t>(t) * p.dense_ld + b] = sv[tk];
                            }
                        } else {
                            const float4 th = *reinterpret_cast<const float4 *>(&sTheta[tl0]);
                            const int4 c4 = *reinterpret_cast<const int4 *>(&sCnt[quarter * TQ + tl0]);
                            const float thv[4] = {th.x, th.y, th.z, th.w};
                            bool pass[4];
                            unsigned m[4];
#pragma unroll
                            for (int tk = 0; tk < 4; ++tk) {
                                const int t = t0 + tl0 + tk;
                                const bool valid = !MASKED || ((t < L32) && (b < (t >> p.bshift)));
                                pass[tk] = valid && (sv[tk] >= thv[tk]);
                            }
                            // a block enters the token's list when s >= its threshold
                            if (__any_sync(0xFFFFFFFFu, pass[0] | pass[1] | pass[2] | pass[3])) {
#pragma unroll
                                for (int tk = 0; tk < 4; ++tk) m[tk] = __ballot_sync(0xFFFFFFFFu, pass[tk]);
                                uint2 *base = sub + static_cast<int64_t>(tl0) * CAP;
                                const int cnt4[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                                for (int tk = 0; tk < 4; ++tk) {
                                    if (m[tk] == 0u) continue;  // warp-uniform
                                    int *cp = &sCnt[quarter * TQ + tl0 + tk];
                                    const int cnt = cnt4[tk];
                                    const int pos = cnt + __popc(m[tk] & ltmask);
                                    st_global_pred(base + tk * CAP + pos,
                                                   make_uint2(__float_as_uint(sv[tk]), static_cast<uint32_t>(b)),
                                                   pass[tk] && pos < SUB);
                                    *cp = cnt + __popc(m[tk]);
                                }
                            }
                        }
                        if (ch + 1 < GTOK / 4) tmem_wait16(curb[(ch + 1) & 1]);
                    }
                };
                if (masked) score_tile(std::true_type{});
                else score_tile(std::false_type{});
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[buf]);
                ++acc;
                if (!check) continue;
                // a sub-list that might overflow within the next CHK tiles gets
                // cut back now (not needed after the last tile)
                const int par = static_cast<int>(nchk & 1);
                ++nchk;
                if (!last) {
                    // a token with many blocks still waiting for its first
                    // prediction is cut back early, so that its threshold
                    // rises before most of its blocks stream past
                    const int tln = g * GTOK + (lane & (GTOK - 1));
                    const bool early = predict_on && sPred[tln] == -INFINITY &&
                                       ((t0 + tln) >> p.bshift) > 8 * static_cast<int64_t>(p.k_sel);
                    const bool full_soon = lane < GTOK && sCnt[quarter * TQ + tln] > (early ? FIRST_AT : FLAG_AT);
                    const unsigned fl = __ballot_sync(0xFFFFFFFFu, full_soon);
                    if (fl && lane == 0) atomicOr(&sFlag[g * 2 + par], fl);
                }
                if (group_sync_fail(bar, sMisc[1] != 0)) { ok = false; break; }
                unsigned flags = last ? 0u : sFlag[g * 2 + par];
                if (flags == 0u) continue;
                while (flags) {
                    const int t16 = __ffs(flags) - 1;
                    flags &= flags - 1;
                    const int tl = g * GTOK + t16;
                    int n[4];
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) n[qq] = sCnt[qq * TQ + tl];
                    if (max(max(n[0], n[1]), max(n[2], n[3])) > SUB && tg == 0)
                        report(p.status, QSA_ERR_DEVICE_CHECK);
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) n[qq] = min(n[qq], SUB);
                    if (n[0] + n[1] + n[2] + n[3] <= p.k_sel) continue;  // nothing to cut (the group agrees)
                    uint2 *lst = p.cand + (static_cast<int64_t>(blockIdx.x) * TQ + tl) * CAP;
                    const int nown = min(sCnt[quarter * TQ + tl], SUB);  // this warp's sub-list
                    uint2 it[IPL];
                    group_load(lst + quarter * SUB, nown, it, lane);
                    // the rank a threshold is predicted from (see below)
                    int64_t rp = 0;
                    if (predict_on) {
                        const int64_t ct = (t0 + tl) >> p.bshift;
                        const int64_t seen = min(static_cast<int64_t>(j + 1) * TB, ct);
                        rp = (MARGIN * static_cast<int64_t>(p.k_sel) * seen + ct - 1) / ct;
                        if (rp < R_MIN) rp = R_MIN;
                    }
                    const bool pred = predict_on && rp < p.k_sel;
                    // cheap pass: a bucket bound 16 bits below the shared prefix
                    // (with the predicted rank's bucket in the same steps)
                    RadixOut r, rq;
                    if (pred) group_radix2(it, nown, p.k_sel, static_cast<int>(rp), G, r, rq);
                    else r = group_radix<false, false>(it, nown, 0u, p.k_sel, 2, G);
                    float th;
                    StagedRule rule{r.thr, 0u, 1};
                    if ((p.k_sel - r.krem) + r.eq <= KEEP_MAX)
                        th = r.lo == 0 ? nextafterf(key2f(r.thr), INFINITY) : key2f(r.thr);
                    else
                        rule = group_select_exact(it, nown, p.k_sel, G, &th);
                    // survivors back to the list (every warp has its items in
                    // registers by now), dealt round-robin over the 4 sub-lists
                    const int kept = group_ranks_apply(
                        it, nown, [&](uint2 e) { return staged_keep(rule, e); },
                        [&](uint2 e, int pos) {
                            lst[(pos & 3) * SUB + (pos >> 2)] = make_uint2(__float_as_uint(key2f(e.x)), e.y);
                        },
                        G);
                    if (tg < 4) sCnt[tg * TQ + tl] = (kept + 3 - tg) / 4;
                    if (tg == 0) sTheta[tl] = th;
                    if (pred) {
                        // Predicted threshold: the rp-th best score seen so far,
                        // rp = 2 (budget-1) seen / c, is expected to keep about
                        // twice the budget of the token's c blocks above it.  It
                        // holds a later block back only if the token's final
                        // (budget-1)-th best reaches it, which finalize checks
                        // against the highest prediction the token ever had: a
                        // later, lower prediction lowers neither (blocks below
                        // the earlier one were already held back).
                        // rq.thr is at or below the rp-th best key (rp < budget-1
                        // <= kept: the list holds at least rp entries)
                        const float thp = fmaxf(sPred[tl], key2f(rq.thr));
                        if (tg == 0) {
                            sPred[tl] = thp;
                            sTheta[tl] = fmaxf(th, thp);
                        }
                    }
                }
                if (group_sync_fail(bar, false)) { ok = false; break; }
                if (tg == 0) sFlag[g * 2 + par] = 0u;  // next written two checks from now
            }
            if (!ok) continue;  // the next tile-start barrier takes everyone out
            if constexpr (!DENSE) {
                // ---- finalize: the group's 16 tokens one after the other
                bool pred_failed = false;
                for (int t16 = 0; t16 < GTOK; ++t16) {
                    const int tl = g * GTOK + t16;
                    const int t = t0 + tl;
                    if (t >= L32) break;
                    const int64_t c = t >> p.bshift;
                    int n[4];
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) n[qq] = min(sCnt[qq * TQ + tl], SUB);
                    const int ntot = n[0] + n[1] + n[2] + n[3];
                    const uint2 *lst = p.cand + (static_cast<int64_t>(blockIdx.x) * TQ + tl) * CAP;
                    const int nown = min(sCnt[quarter * TQ + tl], SUB);  // this warp's sub-list
                    uint2 it[IPL];
                    group_load(lst + quarter * SUB, nown, it, lane);
                    StagedRule rule{0u, 0u, 1};
                    if (ntot > p.k_sel) {
                        float th;
                        rule = group_select_exact(it, nown, p.k_sel, G, &th);
                    }
                    const float pred = sPred[tl];
                    if (pred != -INFINITY) {
                        // exact only if (budget-1) candidates reach the predicted threshold
                        const uint32_t pk = f2key(pred);
                        const int reach = group_count(it, nown, [&](uint2 e) { return e.x >= pk; }, G);
                        pred_failed |= reach < p.k_sel;
                    }
                    auto keep = [&](uint2 e) { return staged_keep(rule, e); };
                    // order by block (blocks are distinct): a group sort of 512 keys,
                    // block indices alone or (block, score bits) when scores are written.
                    // The sort input sits in slots 512.. of the group's sort area; the
                    // sort's own first write goes to slots 0..511 (see group_sort512).
                    int32_t *row = p.idx + (t - p.q_off) * p.budget;
                    float *srow = p.score ? p.score + (t - p.q_off) * p.budget : nullptr;
                    int m;
                    auto emit = [&](int e, uint32_t blk, float sc) {
                        if (e >= p.budget) return;
                        const bool in = e < m;
                        row[e] = in ? static_cast<int32_t>(blk) : (e == m ? static_cast<int32_t>(c) : -1);
                        if (srow) srow[e] = in ? sc : (e == m ? INFINITY : -INFINITY);
                    };
                    if (srow) {
                        m = group_ranks_apply(
                            it, nown, keep,
                            [&](uint2 e, int pos) {
                                if (pos < 512)
                                    sort64[512 + pos] = (static_cast<unsigned long long>(e.y) << 32) |
                                                        __float_as_uint(key2f(e.x));
                            },
                            G);
                        group_bar(bar);
                        if (m > 512) {
                            if (tg == 0) report(p.status, QSA_ERR_DEVICE_CHECK);
                            m = 512;
                        }
                        unsigned long long v[4];
#pragma unroll
                        for (int r = 0; r < 4; ++r) v[r] = 4 * tg + r < m ? sort64[512 + 4 * tg + r] : ~0ull;
                        group_sort512(v, sort64, tg, bar);
#if QSA_DEBUG_CHECKS
                        debug_check(p.status, m == static_cast<int>(c < p.k_sel ? c : p.k_sel));
#pragma unroll
                        for (int r = 0; r < 4; ++r)
                            if (4 * tg + r < m)
                                debug_check(p.status, (v[r] >> 32) < static_cast<uint64_t>(c) &&
                                                          (r == 0 || (v[r - 1] >> 32) < (v[r] >> 32)));
#endif
#pragma unroll
                        for (int r = 0; r < 4; ++r)
                            emit(4 * tg + r, static_cast<uint32_t>(v[r] >> 32),
                                 __uint_as_float(static_cast<uint32_t>(v[r])));
                    } else {
                        m = group_ranks_apply(
                            it, nown, keep,
                            [&](uint2 e, int pos) {
                                if (pos < 512) sort32[512 + pos] = e.y;
                            },
                            G);
                        group_bar(bar);
                        if (m > 512) {
                            if (tg == 0) report(p.status, QSA_ERR_DEVICE_CHECK);
                            m = 512;
                        }
                        uint32_t v[4];
#pragma unroll
                        for (int r = 0; r < 4; ++r) v[r] = 4 * tg + r < m ? sort32[512 + 4 * tg + r] : 0xFFFFFFFFu;
                        group_sort512(v, sort32, tg, bar);
                        const int e0 = 4 * tg;
#if QSA_DEBUG_CHECKS
                        debug_check(p.status, m == static_cast<int>(c < p.k_sel ? c : p.k_sel));
#pragma unroll
                        for (int r = 0; r < 4; ++r)
                            if (e0 + r < m)
                                debug_check(p.status, v[r] < static_cast<uint64_t>(c) && (r == 0 || v[r - 1] < v[r]));
#endif
                        if ((p.budget & 3) == 0 && e0 + 3 < m) {
                            *reinterpret_cast<int4 *>(row + e0) = make_int4(
                                static_cast<int>(v[0]), static_cast<int>(v[1]), static_cast<int>(v[2]),
                                static_cast<int>(v[3]));
                        } else {
#pragma unroll
                            for (int r = 0; r < 4; ++r) emit(e0 + r, v[r], 0.f);
                        }
                    }
                }
                // this group's tokens of the tile: redone without prediction if one failed
                if (p.redo && !p.redo_pass && tg == 0) p.redo[4 * static_cast<int64_t>(q) + g] = pred_failed ? 1 : 0;
                if (pred_failed) {
                    predict_on = false;
                    if (tg == 0) {
                        sMisc[2] = 1u;
                        if (p.stop) *reinterpret_cast<volatile int *>(p.stop) = 1;
                    }
                }
            }
        }
        if (!ok) {
            report(p.status, QSA_ERR_TIMEOUT);
            sMisc[1] = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// Budget 1: only the current block, no scoring at all.
__global__ void fill_current_kernel(int64_t q_off, int64_t Lq, int bshift, int budget, int32_t *idx, float *score) {
    const int64_t total = Lq * budget;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t tl = i / budget;
        const int r = static_cast<int>(i - tl * budget);
        idx[i] = r == 0 ? static_cast<int32_t>((q_off + tl) >> bshift) : -1;
        if (score) score[i] = r == 0 ? INFINITY : -INFINITY;
    }
}

}  // namespace ix

int index_grid(int64_t L, int sms) {
    const int64_t nq = (L + ix::TQ - 1) / ix::TQ;
    return static_cast<int>(nq < sms ? nq : sms);
}

// Candidate lists of the persistent grid, then the per-(query tile, group)
// flags of the predicting pass.
size_t index_cand_bytes(int64_t L, int sms) {
    const int64_t nq = (L + ix::TQ - 1) / ix::TQ;
    const size_t lists = static_cast<size_t>(index_grid(L, sms)) * ix::TQ * ix::CAP * sizeof(uint2);
    return lists + ((static_cast<size_t>(nq) * 4 + 255) / 256) * 256 + 256;  // + the call's stop word
}

cudaError_t launch_index(const CUtensorMap &map_q, const CUtensorMap &map_k, int64_t q_off, int64_t Lq,
                         int unit_tokens, int budget, const uint16_t *w, int32_t *idx, float *score,
                         float *dense, void *cand_ws, int32_t *status, int sms, int *stop,
                         cudaStream_t stream) {
    ix::Params p;
    const int64_t L = q_off + Lq;
    p.L = L;
    p.unit_rows = unit_tokens == 1 ? L : L / kBlock;
    p.q_off = q_off;
    p.bshift = unit_tokens == 1 ? 0 : 2;
    p.nq = static_cast<int>((Lq + ix::TQ - 1) / ix::TQ);
    p.k_sel = budget - 1;
    p.budget = budget;
    p.w = w;
    p.idx = idx;
    p.score = score;
    p.dense = dense;
    p.dense_ld = L / kBlock;
    p.cand = reinterpret_cast<uint2 *>(cand_ws);
    p.status = status;
    const int grid = index_grid(Lq, sms);
    // selection launches predict thresholds; a second launch redoes, without
    // prediction, the query tiles whose prediction failed its check (it finds
    // no flag set and leaves at once in all but rare cases)
    p.predict = dense ? 0 : 1;
    p.redo = dense ? nullptr
                   : reinterpret_cast<uint8_t *>(cand_ws) + static_cast<size_t>(grid) * ix::TQ * ix::CAP * sizeof(uint2);
    p.redo_pass = 0;
    p.stop = stop;
    cudaError_t e;
    if (dense) {
        e = cudaFuncSetAttribute(ix::index_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 ix::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        ix::index_kernel<true><<<grid, ix::THREADS, ix::SMEM_BYTES, stream>>>(map_q, map_k, p);
    } else {
        e = cudaFuncSetAttribute(ix::index_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 ix::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        ix::index_kernel<false><<<grid, ix::THREADS, ix::SMEM_BYTES, stream>>>(map_q, map_k, p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        p.predict = 0;
        p.redo_pass = 1;
        ix::index_kernel<false><<<grid, ix::THREADS, ix::SMEM_BYTES, stream>>>(map_q, map_k, p);
    }
    return cudaGetLastError();
}

cudaError_t launch_fill_current_only(int64_t q_off, int64_t Lq, int unit_tokens, int budget, int32_t *idx,
                                     float *score, cudaStream_t stream) {
    int64_t blocks = (Lq * budget + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    ix::fill_current_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(q_off, Lq, unit_tokens == 1 ? 0 : 2,
                                                                           budget, idx, score);
    return cudaGetLastError();
}

}  // namespace qsa
