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
// Design (one persistent CTA per SM, 12 warps):
//   * the contraction runs "swap-AB": the MMA's M = 128 block keys (A, from a
//     TMA tile of kblk), N = 256 columns = 64 query tokens x 4 indexer heads
//     (B, a TMA tile of qi that stays resident for the whole query tile),
//     K = 128; fp32 accumulators live in TMEM, double-buffered (2 x 256 cols);
//   * warp 0 issues the TMA loads, warp 1 issues tcgen05.mma (one thread),
//     warps 4..11 are the epilogue: each thread owns one TMEM lane = one
//     block, reads the 4 head columns of a token, forms the score and tests it
//     against the token's running threshold;
//   * selection is an exact streaming top-k: every token keeps a candidate
//     list (global workspace, L2-resident) of the blocks that beat its
//     threshold.  When a list fills up, a warp radix-selects its k-th best
//     (score desc, index asc), compacts the list to exactly k entries and
//     raises the threshold to that score.  Block tiles are visited in
//     ascending block order, so a later block with a score equal to the
//     threshold always loses the tie and is never needed;
//   * after the last block tile a warp per token selects the final k, sorts
//     them by block index and writes the row.
#include "qsa_common.cuh"
#include "qsa_kernels.h"
#include "qsa_select.cuh"

namespace qsa {
namespace ix {

constexpr int TQ = 64;               // query tokens per tile
constexpr int NCOL = TQ * kHI;       // 256 MMA columns (token-major, head-minor)
constexpr int TB = 128;              // block keys per block tile (MMA M)
constexpr int NSTAGE = 3;            // kblk tile ring
constexpr int CAP = 1024;            // candidate slots per token (32 per lane)
constexpr int SUB = CAP / 4;         // per-warp sub-list of a token (one per TMEM lane quarter)
constexpr int KSTEPS = kDI / 16;     // 8 MMAs of K = 16
constexpr int NEPI = 8;              // epilogue warps
constexpr int THREADS = (4 + NEPI) * 32;
constexpr int SORTN = 512;           // sort buffer per epilogue warp (>= budget-1)

constexpr uint32_t IDESC = idesc_bf16_f32(TB, NCOL);

constexpr int SQ_BYTES = 2 * NCOL * 128;     // two 64-wide K halves, 128-B rows
constexpr int SK_BYTES = 2 * TB * 128;
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + SQ_BYTES;
constexpr int OFF_SORT = OFF_K + NSTAGE * SK_BYTES;
constexpr int OFF_HIST = OFF_SORT + NEPI * SORTN * 8;
constexpr int OFF_W = OFF_HIST + NEPI * 256 * 4;
constexpr int OFF_THETA = OFF_W + TQ * 4 * 4;
constexpr int OFF_CNT = OFF_THETA + TQ * 4;  // [4 quarters][TQ] sub-list counts
constexpr int OFF_BAR = OFF_CNT + 4 * TQ * 4;
constexpr int NBAR = 2 * NSTAGE + 2 + 4;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack

struct Params {
    int64_t L;
    int nq;
    int k_sel;          // budget - 1
    int budget;
    const uint16_t *w;  // [L, 4]
    int32_t *idx;       // [L, budget]
    float *score;       // [L, budget] or null
    float *dense;       // [L, L/4] (dense mode)
    int64_t dense_ld;
    uint2 *cand;        // [grid, TQ, CAP] {score bits, block}
    int32_t *status;
};

__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ int num_btiles(int64_t L, int q) {
    int64_t t_last = static_cast<int64_t>(q) * TQ + TQ - 1;
    if (t_last > L - 1) t_last = L - 1;
    const int64_t cmax = t_last / kBlock;  // blocks 0..cmax-1 are scored
    return static_cast<int>((cmax + TB - 1) / TB);
}

// A token's candidate list is 4 sub-lists of SUB entries, one per epilogue
// warp of its half (the warp that owns TMEM lane quarter q appends to
// sub-list q with a warp-private count, so appending needs neither atomics
// nor shuffles).  Entries are (score bits, block).  For selection the union
// is loaded into registers as (order-preserving key, block): item i of a
// lane is entry (i % 8) * 32 + lane of sub-list i / 8.
constexpr int NI = CAP / 32;
constexpr int KEEP_MAX = CAP - 2 * TB;  // a lower-bound compaction must keep at most this many

__device__ __forceinline__ uint32_t load_union(const uint2 *lst, const int (&n)[4],
                                               uint32_t (&key)[NI], uint32_t (&blk)[NI], int lane) {
    uint32_t vm = 0;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int q = i >> 3;
        const int e = (i & 7) * 32 + lane;
        uint2 it = make_uint2(0u, 0u);
        if (e < n[q]) {
            it = lst[q * SUB + e];
            vm |= 1u << i;
        }
        key[i] = f2key(__uint_as_float(it.x));
        blk[i] = it.y;
    }
    __syncwarp();  // every lane's reads are done before anyone rewrites the list
    return vm;
}

// Write the items whose bit is set in `sel` back, dealt round-robin over the
// 4 sub-lists; returns the total kept (sub-list q then holds (kept+3-q)/4).
__device__ __forceinline__ int store_union(uint2 *lst, const uint32_t (&key)[NI],
                                           const uint32_t (&blk)[NI], uint32_t sel, int lane) {
    int out = 0;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const bool keep = (sel >> i) & 1u;
        const unsigned ball = __ballot_sync(0xFFFFFFFFu, keep);
        if (keep) {
            const int r = out + __popc(ball & ((1u << lane) - 1u));
            lst[(r & 3) * SUB + (r >> 2)] = make_uint2(__float_as_uint(key2f(key[i])), blk[i]);
        }
        out += __popc(ball);
    }
    return out;
}

template <bool DENSE>
__global__ void __launch_bounds__(THREADS, 1)
    index_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                 Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem + OFF_Q;
    uint8_t *sK = smem + OFF_K;
    unsigned long long *sSort = reinterpret_cast<unsigned long long *>(smem + OFF_SORT);
    uint32_t *sHist = reinterpret_cast<uint32_t *>(smem + OFF_HIST);
    float *sW = reinterpret_cast<float *>(smem + OFF_W);
    float *sTheta = reinterpret_cast<float *>(smem + OFF_THETA);
    int *sCnt = reinterpret_cast<int *>(smem + OFF_CNT);  // sCnt[q * TQ + tl]
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
                const int nbt = num_btiles(p.L, q);
                if (nbt == 0) continue;
                if (!mbar_wait(qempty, qph ^ 1)) { ok = false; break; }
                qph ^= 1;
                mbar_arrive_expect_tx(qfull, SQ_BYTES);
                tma_load_2d(sQ, &map_q, qfull, 0, q * NCOL);
                tma_load_2d(sQ + SQ_BYTES / 2, &map_q, qfull, 64, q * NCOL);
                for (int j = 0; j < nbt; ++j) {
                    if (sMisc[1]) { ok = false; break; }
                    if (!mbar_wait(&empty[st], ph ^ 1)) { ok = false; break; }
                    uint8_t *dst = sK + st * SK_BYTES;
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
                const int nbt = num_btiles(p.L, q);
                if (nbt == 0) continue;
                if (!mbar_wait(qfull, qph)) { ok = false; break; }
                qph ^= 1;
                tc_fence_after();
                for (int j = 0; j < nbt; ++j) {
                    if (sMisc[1]) { ok = false; break; }
                    const uint32_t buf = acc & 1;
                    const uint32_t use = acc >> 1;
                    if (!mbar_wait(&tempty[buf], (use & 1) ^ 1)) { ok = false; break; }
                    if (!mbar_wait(&full[st], ph)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d = tmem_base + buf * NCOL;
#pragma unroll
                    for (int ks = 0; ks < KSTEPS; ++ks) {
                        const uint32_t half = ks >> 2, off = (ks & 3) * 32;
                        const uint64_t ad = sdesc_sw128(sk_addr + st * SK_BYTES + half * (SK_BYTES / 2) + off);
                        const uint64_t bd = sdesc_sw128(sq_addr + half * (SQ_BYTES / 2) + off);
                        tc_mma_bf16(d, ad, bd, IDESC, ks > 0 ? 1u : 0u);
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
        const int e = warp - 4;
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        const int half = e >> 2;       // token half: columns [half*128, half*128+128)
        const int tid_h = quarter * 32 + lane;
        uint32_t *hist = sHist + e * 256;
        unsigned long long *sortb = sSort + e * SORTN;
        const unsigned ltmask = (1u << lane) - 1u;
        // this warp's sub-lists: token tl's at sub[tl * CAP]
        uint2 *sub = p.cand + static_cast<int64_t>(blockIdx.x) * TQ * CAP + quarter * SUB;
        uint32_t acc = 0;
        bool ok = true;
        for (int kk = blockIdx.x; kk < p.nq && ok; kk += gridDim.x) {
            const int q = p.nq - 1 - kk;
            const int64_t t0 = static_cast<int64_t>(q) * TQ;
            const int nbt = num_btiles(p.L, q);
            named_bar(1 + half, 128);
            if (tid_h < 32) {
                const int tl = half * 32 + tid_h;
                const int64_t t = t0 + tl;
#pragma unroll
                for (int q = 0; q < 4; ++q) sCnt[q * TQ + tl] = 0;
                sTheta[tl] = -INFINITY;
#pragma unroll
                for (int h = 0; h < kHI; ++h) {
                    float wv = 0.f;
                    if (t < p.L) wv = __uint_as_float(static_cast<uint32_t>(p.w[t * kHI + h]) << 16);
                    sW[tl * 4 + h] = wv;
                }
            }
            named_bar(1 + half, 128);
            const bool tile_all_in = (t0 + TQ <= p.L);
            const int64_t c_min = t0 / kBlock;
            for (int j = 0; j < nbt; ++j) {
                const uint32_t buf = acc & 1;
                const uint32_t use = acc >> 1;
                if (!mbar_wait(&tfull[buf], use & 1)) { ok = false; break; }
                tc_fence_after();
                const int64_t b = static_cast<int64_t>(j) * TB + quarter * 32 + lane;
                const bool masked = !(tile_all_in && (static_cast<int64_t>(j) * TB + TB <= c_min));
                const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       buf * NCOL + half * 128;
                uint32_t ra[32], rb[32];
                tmem_ld32(tbase, ra);
                tmem_wait32(ra);
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t(&cur)[32] = (ch & 1) ? rb : ra;
                    uint32_t(&nxt)[32] = (ch & 1) ? ra : rb;
                    if (ch < 3) tmem_ld32(tbase + (ch + 1) * 32, nxt);  // overlaps the math below
                    const int tl0 = half * 32 + ch * 8;
                    float th[8];
                    *reinterpret_cast<float4 *>(&th[0]) = *reinterpret_cast<const float4 *>(&sTheta[tl0]);
                    *reinterpret_cast<float4 *>(&th[4]) = *reinterpret_cast<const float4 *>(&sTheta[tl0 + 4]);
                    int cnt8[8];
                    if constexpr (!DENSE) {
                        *reinterpret_cast<int4 *>(&cnt8[0]) = *reinterpret_cast<const int4 *>(&sCnt[quarter * TQ + tl0]);
                        *reinterpret_cast<int4 *>(&cnt8[4]) = *reinterpret_cast<const int4 *>(&sCnt[quarter * TQ + tl0 + 4]);
                    }
#pragma unroll
                    for (int tk = 0; tk < 8; ++tk) {
                        const int tl = tl0 + tk;
                        const float4 wv = *reinterpret_cast<const float4 *>(&sW[tl * 4]);
                        // the first product is added to +0 so the sum is never -0
                        float s = fmaf(wv.x, fmaxf(__uint_as_float(cur[4 * tk + 0]), 0.f), 0.0f);
                        s = fmaf(wv.y, fmaxf(__uint_as_float(cur[4 * tk + 1]), 0.f), s);
                        s = fmaf(wv.z, fmaxf(__uint_as_float(cur[4 * tk + 2]), 0.f), s);
                        s = fmaf(wv.w, fmaxf(__uint_as_float(cur[4 * tk + 3]), 0.f), s);
                        const int64_t t = t0 + tl;
                        bool valid = true;
                        if (masked) valid = (t < p.L) && (b < t / kBlock);
                        if constexpr (DENSE) {
                            if (valid) p.dense[t * p.dense_ld + b] = s;
                        } else {
                            // a block enters the token's list when s >= its threshold:
                            // position from a ballot, no branch, no atomic
                            const bool pass = valid && (s >= th[tk]);
                            const unsigned m = __ballot_sync(0xFFFFFFFFu, pass);
                            const int pos = cnt8[tk] + __popc(m & ltmask);
                            if (pass && pos < SUB)
                                sub[static_cast<int64_t>(tl) * CAP + pos] =
                                    make_uint2(__float_as_uint(s), static_cast<uint32_t>(b));
                            cnt8[tk] += __popc(m);
                        }
                    }
                    if constexpr (!DENSE) {
                        *reinterpret_cast<int4 *>(&sCnt[quarter * TQ + tl0]) = *reinterpret_cast<const int4 *>(&cnt8[0]);
                        *reinterpret_cast<int4 *>(&sCnt[quarter * TQ + tl0 + 4]) = *reinterpret_cast<const int4 *>(&cnt8[4]);
                    }
                    if (ch < 3) tmem_wait32(nxt);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[buf]);
                ++acc;
                if constexpr (!DENSE) {
                    // lists that might overflow on the next tile are cut back
                    named_bar(1 + half, 128);
                    for (int i = 0; i < 8; ++i) {
                        const int tl = half * 32 + quarter + 4 * i;
                        int n[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) n[q] = sCnt[q * TQ + tl];
                        const int nmax = max(max(n[0], n[1]), max(n[2], n[3]));
                        if (nmax > SUB) report(p.status, QSA_ERR_DEVICE_CHECK);
                        if (nmax > SUB - 32) {
#pragma unroll
                            for (int q = 0; q < 4; ++q) n[q] = min(n[q], SUB);
                            uint2 *lst = p.cand + (static_cast<int64_t>(blockIdx.x) * TQ + tl) * CAP;
                            uint32_t key[NI], blk[NI];
                            const uint32_t vm = load_union(lst, n, key, blk, lane);
                            // cheap pass: a bucket bound 16 bits below the shared prefix
                            const RadixOut r = warp_radix<NI>(key, vm, p.k_sel, 2, hist, lane);
                            uint32_t sel = 0;
                            float th;
                            if ((p.k_sel - r.krem) + r.eq <= KEEP_MAX) {
#pragma unroll
                                for (int q2 = 0; q2 < NI; ++q2)
                                    if (((vm >> q2) & 1u) && key[q2] >= r.thr) sel |= 1u << q2;
                                th = r.lo == 0 ? nextafterf(key2f(r.thr), INFINITY) : key2f(r.thr);
                            } else {
                                sel = warp_select_exact<NI>(key, blk, vm, p.k_sel, hist, lane, &th);
                            }
                            const int kept = store_union(lst, key, blk, sel, lane);
                            if (lane < 4) sCnt[lane * TQ + tl] = (kept + 3 - lane) / 4;
                            if (lane == 0) sTheta[tl] = th;
                            __syncwarp();
                        }
                    }
                    named_bar(1 + half, 128);
                }
                if (sMisc[1]) { ok = false; break; }
            }
            if (!ok) break;
            if constexpr (!DENSE) {
                // ---- finalize: one warp per token
                for (int i = 0; i < 8; ++i) {
                    const int tl = half * 32 + quarter + 4 * i;
                    const int64_t t = t0 + tl;
                    if (t >= p.L) continue;
                    const int64_t c = t / kBlock;
                    int nq4[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) nq4[q] = min(sCnt[q * TQ + tl], SUB);
                    const int n = nq4[0] + nq4[1] + nq4[2] + nq4[3];
                    const uint2 *lst = p.cand + (static_cast<int64_t>(blockIdx.x) * TQ + tl) * CAP;
                    uint32_t key[NI], blk[NI];
                    const uint32_t vm = load_union(lst, nq4, key, blk, lane);
                    uint32_t sel = vm;
                    if (n > p.k_sel) {
                        float th;
                        sel = warp_select_exact<NI>(key, blk, vm, p.k_sel, hist, lane, &th);
                    }
                    // the kept items as (block << 32 | score bits), sorted by block
                    int m = 0;
#pragma unroll
                    for (int q2 = 0; q2 < NI; ++q2) {
                        const bool keep = (sel >> q2) & 1u;
                        const unsigned ball = __ballot_sync(0xFFFFFFFFu, keep);
                        if (keep) {
                            const int pos = m + __popc(ball & ((1u << lane) - 1u));
                            if (pos < SORTN)
                                sortb[pos] = (static_cast<unsigned long long>(blk[q2]) << 32) |
                                             __float_as_uint(key2f(key[q2]));
                        }
                        m += __popc(ball);
                    }
                    if (m > SORTN) { report(p.status, QSA_ERR_DEVICE_CHECK); m = SORTN; }
                    int P2 = 32;
                    while (P2 < m) P2 <<= 1;
                    for (int ii = m + lane; ii < P2; ii += 32) sortb[ii] = ~0ull;
                    __syncwarp();
                    for (int kb = 2; kb <= P2; kb <<= 1) {
                        for (int jb = kb >> 1; jb > 0; jb >>= 1) {
                            for (int ii = lane; ii < P2; ii += 32) {
                                const int ix = ii ^ jb;
                                if (ix > ii) {
                                    const unsigned long long a = sortb[ii], bb = sortb[ix];
                                    const bool up = (ii & kb) == 0;
                                    if ((a > bb) == up) {
                                        sortb[ii] = bb;
                                        sortb[ix] = a;
                                    }
                                }
                            }
                            __syncwarp();
                        }
                    }
                    int32_t *row = p.idx + t * p.budget;
                    float *srow = p.score ? p.score + t * p.budget : nullptr;
                    for (int ii = lane; ii < p.budget; ii += 32) {
                        int32_t bi;
                        float sv;
                        if (ii < m) {
                            const unsigned long long v = sortb[ii];
                            bi = static_cast<int32_t>(v >> 32);
                            sv = __uint_as_float(static_cast<uint32_t>(v));
                        } else if (ii == m) {
                            bi = static_cast<int32_t>(c);
                            sv = INFINITY;
                        } else {
                            bi = -1;
                            sv = -INFINITY;
                        }
                        row[ii] = bi;
                        if (srow) srow[ii] = sv;
                    }
                    __syncwarp();
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
__global__ void fill_current_kernel(int64_t L, int budget, int32_t *idx, float *score) {
    const int64_t total = L * budget;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / budget;
        const int r = static_cast<int>(i - t * budget);
        idx[i] = r == 0 ? static_cast<int32_t>(t / kBlock) : -1;
        if (score) score[i] = r == 0 ? INFINITY : -INFINITY;
    }
}

}  // namespace ix

int index_grid(int64_t L, int sms) {
    const int64_t nq = (L + ix::TQ - 1) / ix::TQ;
    return static_cast<int>(nq < sms ? nq : sms);
}

size_t index_cand_bytes(int64_t L, int sms) {
    return static_cast<size_t>(index_grid(L, sms)) * ix::TQ * ix::CAP * sizeof(uint2);
}

cudaError_t launch_index(const CUtensorMap &map_q, const CUtensorMap &map_k, int64_t L,
                         int budget, const uint16_t *w, int32_t *idx, float *score,
                         float *dense, void *cand_ws, int32_t *status, int sms,
                         cudaStream_t stream) {
    ix::Params p;
    p.L = L;
    p.nq = static_cast<int>((L + ix::TQ - 1) / ix::TQ);
    p.k_sel = budget - 1;
    p.budget = budget;
    p.w = w;
    p.idx = idx;
    p.score = score;
    p.dense = dense;
    p.dense_ld = L / kBlock;
    p.cand = reinterpret_cast<uint2 *>(cand_ws);
    p.status = status;
    const int grid = index_grid(L, sms);
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
    }
    return cudaGetLastError();
}

cudaError_t launch_fill_current_only(int64_t L, int budget, int32_t *idx, float *score,
                                     cudaStream_t stream) {
    int64_t blocks = (L * budget + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    ix::fill_current_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(L, budget, idx, score);
    return cudaGetLastError();
}

}  // namespace qsa
