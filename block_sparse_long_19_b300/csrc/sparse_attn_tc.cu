// Block-sparse GQA attention on the 5th-generation tensor cores (tcgen05,
// TMEM accumulators, TMA-fed), prefill and the split-KV decode step.
//
// What it computes (Qwen3.8-Flash-Next launch post, "Model Architecture /
// Attention: GDN + QSA": attention runs only over the regions the indexer
// selected; model card "Model Overview / Qwen Sparse Attention": 24 query
// heads, 2 KV heads, head dim 256, rotary dim 64): for a query at position t,
// the keys are j with floor(j/4) selected and j <= t; query head h reads KV
// head h/12; O = softmax(Q'K'^T * scale) V with Q' the query after RoPE.
// The same computation as the warp-MMA kernel of sparse_attn.cu, with its
// contractions issued to the tensor cores by one thread.
//
// Data path.  A selected block's 4 key rows of both KV heads (4 KiB of K,
// 4 KiB of V) arrive as ONE 5-D TMA box each, {64 dims, 4 tokens, 2 heads,
// 4 dim chunks, 1 sequence} with the dim-chunk outermost, so the box lands
// as four 1 KiB 128-byte-swizzled atoms: atom c holds dims 64c..64c+63 of the
// 8 rows (head g, token i) in the order 4g + i.  Sixteen blocks make a tile
// (64 KiB of K or of V) whose 128 rows (block, head, token) are the MMA's
// M dimension:
//   * S^T = K Q'^T: A = the K tile, K-major (8-row groups 4 KiB apart),
//     B = Q' (24 heads + 8 unused rows, K-major), M = 128, N = 32, K = 256,
//     fp32 in TMEM (row r of the tile in lane r, column = query head);
//   * O^T += V^T P^T: A = the V tile read MN-major (M = 128 head dims per
//     MMA, two MMAs for the 256; K = the tile's 128 rows), B = P^T in shared
//     memory, MN-major (64-byte swizzle), N = 32 query heads; O^T stays in
//     TMEM for the whole key loop.
// The ring of 3 slots of 64 KiB takes K_0, V_0, K_1, V_1, ... in turn, and a
// slot is refilled as soon as its MMA has read it.
// Every key row meets all 24 query heads in the MMA; the softmax gives
// probability 0 to the 12 heads of the other KV head, so their products
// vanish in PV (half the tensor work is spent on those zeros: the kernel is
// bound by the gather, at about 12 flop per byte, not by the tensor cores).
//
// Softmax.  A thread owns one TMEM lane = one key row and the 12 query heads
// of its KV head.  All rows of a query head need one common reference
// maximum m; it is the exact column maximum of the query's first tile, and
// later tiles keep it unless a score exceeds it by 2^32 (then the column
// maxima of that tile are taken, O^T in TMEM and the partial sums are
// rescaled).  p = 2^(x - m) in fp32, rounded to bf16 for PV (as the warp-MMA
// kernel does); the row sums stay per thread and are added up at the end.
//
// Warp roles (one query (or decode split) per CTA):
//   warps 0-3: softmax (TMEM lane quarter = warp % 4), then the output;
//   warp 4: MMA issuer (one thread): QK^T and PV of the tiles in order, each
//     as soon as its inputs are ready;
//   warp 5: TMEM allocation, Q' (RoPE) into shared memory;
//   warps 6..6+NPROD-1: TMA producers.  Every producer warp issues its share
//     of the 16 block copies of every tile: one warp issues a 4 KiB copy
//     only about every 100 cycles (tensor box or plain bulk copy alike,
//     about 39 GB/s per SM), and the next tile's load cannot start before
//     the ring frees a slot, so a tile's copies are spread over warps.
// Every wait is bounded and also gives up once another warp has reported a
// problem; nothing traps.
#include "qsa_common.cuh"
#include "qsa_kernels.h"

#ifndef QSA_TC_PRODUCERS
#define QSA_TC_PRODUCERS 3
#endif

namespace qsa {
namespace tca {

constexpr int TBLK = 16;                    // selected blocks per tile
constexpr int TROWS = TBLK * 8;             // 128 MMA rows (block x KV head x token)
constexpr int TILE_BYTES = TBLK * 4096;     // K (or V) of a tile: 64 KiB
constexpr int NSLOT = 3;                    // ring slots (K and V tiles alternate)
constexpr int NS = 32;                      // MMA N: 24 query heads + 8 unused
constexpr int Q_PLANE = 3 * 1024;           // one 64-dim chunk of the 24 query rows
constexpr int P_BYTES = TROWS * 64;         // P^T of one tile: 128 rows x 32 bf16
constexpr int P_AREA = 2 * P_BYTES;         // two P^T buffers; they first hold the raw query row
static_assert(2 * P_BYTES <= P_AREA, "P buffers");

constexpr int OFF_RING = 0;
constexpr int OFF_Q = OFF_RING + NSLOT * TILE_BYTES;   // 196608
constexpr int OFF_P = OFF_Q + 4 * Q_PLANE;             // the 4th row group of chunk 3 reads P's first KiB
constexpr int OFF_IDX = OFF_P + P_AREA;
constexpr int OFF_RED = OFF_IDX + kMaxBudget * 4;      // [4 warps][32] u32
constexpr int OFF_LSUM = OFF_RED + 4 * 32 * 4;         // [4 warps][2 heads][12] f32
constexpr int OFF_HEAD = OFF_LSUM + 4 * 2 * 12 * 4;    // [3][24] f32 per query head
constexpr int OFF_CS = OFF_HEAD + 3 * 24 * 4;          // cos/sin of the query position
constexpr int OFF_BAR = OFF_CS + 64 * 4;
constexpr int NBAR = 2 * NSLOT + 8 + 3;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM_USED = OFF_MISC + 64;
constexpr int SMEM_BYTES = SMEM_USED + 1024;           // + alignment of the base to 1 KiB
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
static_assert(OFF_Q % 1024 == 0 && OFF_P % 1024 == 0, "swizzle atoms need 1 KiB alignment");

constexpr int NPROD = QSA_TC_PRODUCERS;  // producer warps
constexpr int WARP_MMA = 4, WARP_Q = 5, WARP_PROD = 6;
constexpr int THREADS = (WARP_PROD + NPROD) * 32;
constexpr uint32_t TMEM_COLS = 128;   // S^T: 2 x 32 columns, O^T: 2 halves x 32 columns
constexpr uint32_t COL_O = 64;

// kind::f16 instruction descriptor: D fp32, A and B bf16, A / B MN-major
// flags (bits 15 / 16), N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
           (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}
constexpr uint32_t IDESC_QK = idesc(TROWS, NS, 0, 0);
constexpr uint32_t IDESC_PV = idesc(128, NS, 1, 1);

// Shared-memory matrix descriptor: start >> 4, leading / stride byte
// offsets >> 4, version 1, layout (2 = 128-byte swizzle, 4 = 64-byte).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(layout) << 61);
}

__device__ __forceinline__ void tma_load_5d(void *dst, const CUtensorMap *map, uint64_t *bar, int row, int seq,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(0), "r"(row), "r"(0), "r"(0), "r"(seq),
        "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Non-blocking test of an mbarrier phase (never suspends the thread).
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait that also gives up once the CTA's abort flag is set.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile uint32_t *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (unsigned n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 15u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > kWaitLimitNs) return false;
        }
    }
}

__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Barrier of the 128 softmax threads that also ORs a flag over them.
__device__ __forceinline__ bool softmax_bar_or(bool v) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1 : 0)
        : "memory");
    return r != 0;
}

template <bool DECODE>
__global__ void __launch_bounds__(THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                   AttnArgs a, RopeFreqs f, int64_t key_rows) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sRing = smem + OFF_RING;
    uint8_t *sQ = smem + OFF_Q;
    uint8_t *sP = smem + OFF_P;
    int32_t *sIdx = reinterpret_cast<int32_t *>(smem + OFF_IDX);
    uint32_t *sRed = reinterpret_cast<uint32_t *>(smem + OFF_RED);
    float *sLsum = reinterpret_cast<float *>(smem + OFF_LSUM);
    float *sHead = reinterpret_cast<float *>(smem + OFF_HEAD);
    float *sCS = reinterpret_cast<float *>(smem + OFF_CS);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint64_t *kv_full = bars;
    uint64_t *kv_empty = bars + NSLOT;
    uint64_t *s_full = bars + 2 * NSLOT;      // [2]
    uint64_t *s_empty = s_full + 2;           // [2]
    uint64_t *p_full = s_full + 4;            // [2]
    uint64_t *p_empty = s_full + 6;           // [2]
    uint64_t *q_full = s_full + 8;
    uint64_t *o_full = s_full + 9;
    uint64_t *q_stage = s_full + 10;          // the raw query row, copied into sP
    volatile uint32_t *sMisc = reinterpret_cast<volatile uint32_t *>(smem + OFF_MISC);
    // sMisc[0] TMEM base, sMisc[1] abort flag, sMisc[2] softmax failure flag

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ------------------------------------------------------ work item --
    int64_t t, orow_id;
    int s = 0, split = 0;
    const uint16_t *qrow;
    const int32_t *irow;
    if constexpr (DECODE) {
        s = blockIdx.y;
        split = blockIdx.x;
        const int64_t T = a.seq_lens[s];
        if (T < 1 || T > a.seq_stride) {
            if (threadIdx.x == 0) report(a.status, QSA_ERR_DEVICE_CHECK);
            return;
        }
        t = T - 1;
        orow_id = s;
        qrow = a.q + static_cast<int64_t>(s) * kHQ * kD;
        irow = a.idx + static_cast<int64_t>(s) * a.budget;
    } else {
        orow_id = a.L - 1 - blockIdx.x;
        t = a.q_off + orow_id;
        qrow = a.q + orow_id * (kHQ * kD);
        irow = a.idx + orow_id * a.budget;
    }
    const int64_t c = t / kBlock;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(&kv_full[i], NPROD);
            mbar_init(&kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 4);
            mbar_init(&p_full[i], 4);
            mbar_init(&p_empty[i], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(o_full, 1);
        sMisc[1] = 0;
        sMisc[2] = 0;
        fence_barrier_init();
    }
    if (warp == WARP_Q) {
        // the query row (24 x 256 bf16, 12 KiB) lands in the P buffers, unused
        // until the first probabilities exist (which need Q' first)
        if (lane == 0) {
            mbar_init(q_stage, 1);
            fence_barrier_init();
            mbar_arrive_expect_tx(q_stage, kHQ * kD * 2);
            bulk_g2s(sP, qrow, kHQ * kD * 2, q_stage);
        }
        __syncwarp();  // tcgen05.alloc is warp-collective: the warp must have reconverged
        tmem_alloc(const_cast<uint32_t *>(&sMisc[0]), TMEM_COLS);
        tmem_relinquish();
    }
    if constexpr (DECODE) {
        pdl_trigger();
        pdl_wait();  // the selection written by the decode indexer
    }
    for (int i = threadIdx.x; i < a.budget; i += THREADS) {
        int b = irow[i];
#if QSA_DEBUG_CHECKS
        {  // a row as the indexer writes it: past blocks ascending, block c last, -1 padding
            const int nxt = i + 1 < a.budget ? irow[i + 1] : -1;
            bool row_ok = b >= -1 && b <= c && (i > 0 || b >= 0);
            if (b >= 0) row_ok = row_ok && (nxt < 0 ? b == c : b < nxt);
            else row_ok = row_ok && nxt < 0;
            debug_check(a.status, row_ok);
        }
#endif
        if (b < 0 || b > c) b = -1;  // out-of-range entries are ignored
        sIdx[i] = b;
    }
    if (warp == WARP_Q) {
        float cs, sn;
        rope_cos_sin(t, f.inv_freq[lane], cs, sn);
        sCS[lane] = cs;
        sCS[32 + lane] = sn;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sMisc[0];

    // used slots (the last selected entry + 1) and this CTA's tiles
    int nslot = 0;
    for (int base = 0; base < a.budget; base += 32) {
        const int i = base + lane;
        const unsigned ball = __ballot_sync(0xFFFFFFFFu, i < a.budget && sIdx[i] >= 0);
        if (ball) nslot = base + 32 - __clz(ball);
    }
    const int total = (nslot + TBLK - 1) / TBLK;
    int tb = 0, te = total;
    if constexpr (DECODE) {
        const int per = (total + a.nsplit - 1) / a.nsplit;
        tb = min(total, split * per);
        te = min(total, tb + per);
    }
    const int nt = te - tb;
    volatile uint32_t *abort_flag = &sMisc[1];

    if (warp >= WARP_PROD) {
        // ------------------------------------------------ producers --
        // loads n = 0, 1, 2, ... are K_0, V_0, K_1, V_1, ... into slot n % 3;
        // producer warp w copies blocks w, w + NPROD, ... of each (one per
        // lane) and arrives on the slot's barrier with its byte count.  An
        // unused slot (no block, or beyond the budget) reads rows past the
        // end of the tensor, which TMA fills with zeros (no memory traffic).
        const int pw = warp - WARP_PROD;
        const int mine = (TBLK - pw + NPROD - 1) / NPROD;  // blocks this warp copies per tile
        const uint64_t pol = policy_evict_first();
        const int seq = DECODE ? s : 0;
        const int oob = static_cast<int>(key_rows);
        bool ok = true;
        for (int n = 0; n < 2 * nt; ++n) {
            const int slot = n % NSLOT;
            const int u = n >> 1, kv = n & 1;
            const int j = tb + u;
            if (lane == 0) ok = wait_or_abort(&kv_empty[slot], ((n / NSLOT) & 1) ^ 1, abort_flag);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            if (lane == 0) mbar_arrive_expect_tx(&kv_full[slot], mine * 4096);
            __syncwarp();
            const int blk = pw + NPROD * lane;
            if (lane < mine) {
                const int si = j * TBLK + blk;
                const int b = si < a.budget ? sIdx[si] : -1;
                const int row = b >= 0 ? b * kBlock : oob;
                tma_load_5d(sRing + slot * TILE_BYTES + blk * 4096, kv ? &map_v : &map_k, &kv_full[slot], row,
                            seq, pol);
            }
        }
        // nothing may land in shared memory after the CTA has left: wait for
        // the last loads (normal runs find them complete)
        if (lane == 0 && ok) {
            for (int n = max(0, 2 * nt - NSLOT); n < 2 * nt; ++n)
                if (!mbar_wait(&kv_full[n % NSLOT], (n / NSLOT) & 1)) ok = false;
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok && lane == 0) {
            report(a.status, QSA_ERR_TIMEOUT);
            *abort_flag = 1;
        }
    } else if (warp == WARP_MMA) {
        // ----------------------------------------------- MMA issuer --
        if (lane == 0) {
            bool ok = wait_or_abort(q_full, 0, abort_flag);
            const uint32_t ring = smem_u32(sRing), q_addr = smem_u32(sQ), p_addr = smem_u32(sP);
            // QK^T of tile u needs K_u landed and S buffer u % 2 free (read by
            // the softmax of tile u - 2); PV of tile u needs P_u and V_u.  The
            // two streams are issued in whatever order they become ready, PV
            // first: a PV frees a ring slot for the next loads, so it must not
            // wait behind a QK^T whose K tile is still in flight.  A parity
            // test of a slot's barrier is only meaningful once the slot's
            // previous load has landed.  With the odd ring of 3 slots, K_u
            // goes into the slot of V_{u-2}: QK^T of tile u may only be
            // tested once PV of tile u-2 has been issued (QK^T stays less
            // than two tiles ahead of PV), or the test would read the parity
            // of a phase two behind and pass too early.
            auto issue_qk = [&](int u) {
                const int slot = (2 * u) % NSLOT;
                tc_fence_after();
                const uint32_t d = tmem + (u & 1) * NS;
                const uint32_t kt = ring + slot * TILE_BYTES;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_bf16(d, sdesc(kt + ch * 1024 + kk * 32, 16, 4096, 2),
                                    sdesc(q_addr + ch * Q_PLANE + kk * 32, 16, 1024, 2), IDESC_QK,
                                    (ch | kk) ? 1u : 0u);
                tc_commit(&s_full[u & 1]);
                tc_commit(&kv_empty[slot]);
            };
            auto issue_pv = [&](int u) {
                const int slot = (2 * u + 1) % NSLOT;
                tc_fence_after();
                const uint32_t vt = ring + slot * TILE_BYTES;
                const uint32_t pt = p_addr + (u & 1) * P_BYTES;
#pragma unroll
                for (int kk = 0; kk < TROWS / 16; ++kk)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        tc_mma_bf16(tmem + COL_O + h * NS, sdesc(vt + kk * 8192 + h * 2048, 1024, 4096, 2),
                                    sdesc(pt + kk * 1024, 16, 512, 4), IDESC_PV, (u > 0 || kk > 0) ? 1u : 0u);
                tc_commit(&p_empty[u & 1]);
                tc_commit(&kv_empty[slot]);
            };
            int uq = 0, up = 0;  // next tile for QK^T, next tile for PV
            unsigned long long t0 = globaltimer();
            unsigned spins = 0;
            while (ok && up < nt) {
                if (up < uq && mbar_test(&p_full[up & 1], (up >> 1) & 1) &&
                    mbar_test(&kv_full[(2 * up + 1) % NSLOT], ((2 * up + 1) / NSLOT) & 1)) {
                    issue_pv(up++);
                    t0 = globaltimer();
                    continue;
                }
                if (uq < nt && (NSLOT % 2 == 0 || uq < up + 2) &&
                    mbar_test(&kv_full[(2 * uq) % NSLOT], ((2 * uq) / NSLOT) & 1) &&
                    mbar_test(&s_empty[uq & 1], ((uq >> 1) & 1) ^ 1)) {
                    issue_qk(uq++);
                    t0 = globaltimer();
                    continue;
                }
                if ((++spins & 15u) == 0 && (*abort_flag || globaltimer() - t0 > kWaitLimitNs)) ok = false;
            }
            // o_full completes once every MMA issued here has: the softmax
            // warps read O^T after it, and this thread waits for it too, so no
            // MMA is in flight when the CTA releases TMEM
            tc_commit(o_full);
            if (!mbar_wait(o_full, 0)) ok = false;
            if (!ok) {
                report(a.status, QSA_ERR_TIMEOUT);
                *abort_flag = 1;
            }
        }
    } else if (warp == WARP_Q) {
        // ------------------------------------------- Q' into shared memory --
        // row n (query head) of 64-dim chunk ch at sQ + ch * Q_PLANE + (n/8) KiB
        // + (n%8) * 128, 16-byte piece p stored at p ^ (n % 8) (128-byte swizzle);
        // the raw row is read from its copy in sP
        const int qt = lane;
        const bool staged = mbar_wait(q_stage, 0);  // the copy always lands: no early exit
        const uint16_t *qs = reinterpret_cast<const uint16_t *>(sP);
        auto qdst = [&](int n, int ch, int p) {
            return sQ + ch * Q_PLANE + (n >> 3) * 1024 + (n & 7) * 128 + ((p ^ (n & 7)) << 4);
        };
        for (int i = qt; staged && i < kHQ * 4; i += 32) {  // rotary pieces: dims 8p.. and 32+8p..
            const int n = i >> 2, p = i & 3;
            const uint4 x1v = *reinterpret_cast<const uint4 *>(qs + n * kD + 8 * p);
            const uint4 x2v = *reinterpret_cast<const uint4 *>(qs + n * kD + 32 + 8 * p);
            const uint16_t *x1 = reinterpret_cast<const uint16_t *>(&x1v);
            const uint16_t *x2 = reinterpret_cast<const uint16_t *>(&x2v);
            uint4 y1v, y2v;
            uint16_t *y1 = reinterpret_cast<uint16_t *>(&y1v);
            uint16_t *y2 = reinterpret_cast<uint16_t *>(&y2v);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int r = 8 * p + e;
                const float a1 = __uint_as_float(static_cast<uint32_t>(x1[e]) << 16);
                const float a2 = __uint_as_float(static_cast<uint32_t>(x2[e]) << 16);
                const float cs = sCS[r], sn = sCS[32 + r];
                const __nv_bfloat16 b1 = __float2bfloat16_rn(fmaf(a1, cs, -a2 * sn));
                const __nv_bfloat16 b2 = __float2bfloat16_rn(fmaf(a2, cs, a1 * sn));
                y1[e] = *reinterpret_cast<const uint16_t *>(&b1);
                y2[e] = *reinterpret_cast<const uint16_t *>(&b2);
            }
            *reinterpret_cast<uint4 *>(qdst(n, 0, p)) = y1v;
            *reinterpret_cast<uint4 *>(qdst(n, 0, p + 4)) = y2v;
        }
        for (int i = qt; staged && i < kHQ * 24; i += 32) {  // dims 64..255 unchanged
            const int n = i / 24, r = i % 24, ch = 1 + r / 8, p = r % 8;
            *reinterpret_cast<uint4 *>(qdst(n, ch, p)) = *reinterpret_cast<const uint4 *>(qs + n * kD + ch * 64 + p * 8);
        }
        if (!staged && qt == 0) {
            report(a.status, QSA_ERR_TIMEOUT);
            *abort_flag = 1;
        }
        fence_proxy_async();
        __syncwarp();
        if (qt == 0 && staged) mbar_arrive(q_full);
    } else {
        // ---------------------------------------------------- softmax --
        const int quarter = warp & 3;
        // S^T of a 128-row tile: row r sits in TMEM lane r, so each thread
        // owns one row; O^T (128 lanes) is read the same way
        const bool has_row = true;
        const int r = quarter * 32 + lane;          // tile row of this lane
        const int g = (r >> 2) & 1;                 // KV head of the row
        const int ti = r & 3;                       // token within the block
        const int bl = r >> 3;                      // block within the tile
        const int dr = quarter * 32 + lane;         // O^T lane: head dim dr (and 128 + dr)
        const int tid = threadIdx.x;                // 0..127
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const int64_t t_in_c = t - c * kBlock;      // rows 0..t_in_c of block c are visible
        // per query head (shared): the reference maximum, the last rescale
        // factor, and at the end 1 / row sum; registers hold this row's 12 heads
        float *sM = sHead;
        float *sAlpha = sHead + 24;
        float *sInv = sHead + 48;
        float mm[12], l[12];
#pragma unroll
        for (int n = 0; n < 12; ++n) {
            mm[n] = 0.f;
            l[n] = 0.f;
        }
        bool ok = true;
        // P^T row r: (r/8) * 512 + (r%8) * 64 bytes, 16-byte piece k at k ^ ((r%8)/2)
        const int prow = (r >> 3) * 512 + (r & 7) * 64;
        const int pswz = (r & 7) >> 1;
        // Failures: every wait result is made warp-uniform at once (TMEM loads
        // and stores are warp-collective), and the four warps agree at the
        // per-tile vote: a thread that met one writes sFail before the vote,
        // and after it every thread reads the same value and leaves together.
        volatile uint32_t *sFail = &sMisc[2];
        for (int u = 0; u < nt; ++u) {
            const int j = tb + u;
            ok = __all_sync(0xFFFFFFFFu, ok && wait_or_abort(&s_full[u & 1], (u >> 1) & 1, abort_flag));
            uint32_t v[32];
            if (ok) {
                tc_fence_after();
                tmem_ld32(lane_addr + (u & 1) * NS, v);
                tmem_wait32(v);
            } else {
#pragma unroll
                for (int n = 0; n < 32; ++n) v[n] = 0u;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[u & 1]);
            const int si = j * TBLK + bl;
            const int b = si < a.budget ? sIdx[si] : -1;
            const bool valid = has_row && ok && b >= 0 && (b < c || ti <= t_in_c);
            float x[12];
#pragma unroll
            for (int n = 0; n < 12; ++n)
                x[n] = valid ? __uint_as_float(g ? v[12 + n] : v[n]) * a.scale_log2 : -INFINITY;
            bool over = u == 0;
#pragma unroll
            for (int n = 0; n < 12; ++n) over |= x[n] > mm[n] + 32.f;
            if (!ok) *sFail = 1u;
            const bool vote = softmax_bar_or(over || !ok);
            if (vote && *sFail) break;  // the same decision in all 128 threads
            if (vote) {
                // new reference maxima: the tile's column maxima (first tile),
                // or the larger of those and the old reference
                uint32_t key[12];
#pragma unroll
                for (int n = 0; n < 12; ++n) key[n] = valid ? f2key(x[n]) : 0u;
#pragma unroll
                for (int gg = 0; gg < 2; ++gg)
#pragma unroll
                    for (int n = 0; n < 12; ++n) {
                        const uint32_t kv = __reduce_max_sync(0xFFFFFFFFu, g == gg ? key[n] : 0u);
                        if (lane == 0) sRed[quarter * 32 + gg * 12 + n] = kv;
                    }
                named_bar(1, 128);
                if (tid < 24) {
                    const uint32_t k = max(max(sRed[tid], sRed[32 + tid]), max(sRed[64 + tid], sRed[96 + tid]));
                    const float mx = k == 0u ? -INFINITY : key2f(k);
                    const float mold = u == 0 ? 0.f : sM[tid];
                    const float mnew = u == 0 ? (mx == -INFINITY ? 0.f : mx) : fmaxf(mold, mx);
                    sAlpha[tid] = u == 0 ? 1.f : exp2f(mold - mnew);
                    sM[tid] = mnew;
                }
                named_bar(1, 128);
#pragma unroll
                for (int n = 0; n < 12; ++n) {
                    mm[n] = sM[12 * g + n];
                    l[n] *= sAlpha[12 * g + n];
                }
                if (u > 0) {
                    // O^T holds the sums of tiles 0..u-1 once PV of tile u-1 is done
                    ok = __all_sync(0xFFFFFFFFu,
                                    wait_or_abort(&p_empty[(u - 1) & 1], ((u - 1) >> 1) & 1, abort_flag));
                    if (ok) {
                        tc_fence_after();
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t o[32];
                            tmem_ld32(lane_addr + COL_O + h * NS, o);
                            tmem_wait32(o);
#pragma unroll
                            for (int n = 0; n < 24; ++n) o[n] = __float_as_uint(__uint_as_float(o[n]) * sAlpha[n]);
                            tmem_st32(lane_addr + COL_O + h * NS, o);
                        }
                        tmem_wait_st();
                    }
                }
            }
            // probabilities of this row for its KV head's 12 query heads
            uint32_t pk[6];
#pragma unroll
            for (int n = 0; n < 12; n += 2) {
                const float p0 = exp2f(x[n] - mm[n]);
                const float p1 = exp2f(x[n + 1] - mm[n + 1]);
                l[n] += p0;
                l[n + 1] += p1;
                pk[n / 2] = pack_bf16(p0, p1);
            }
            // the block of position t: rows after t must not reach PV, even as
            // 0 * (whatever the cache holds there): zero them in the V tile
            if (has_row && ok && b == c && ti > t_in_c) {
                const int n = 2 * u + 1, slot = n % NSLOT;
                if (!wait_or_abort(&kv_full[slot], (n / NSLOT) & 1, abort_flag)) ok = false;
                if (ok) {
                    uint8_t *vrow = sRing + slot * TILE_BYTES + bl * 4096 + (4 * g + ti) * 128;
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch)
#pragma unroll
                        for (int p = 0; p < 8; ++p)
                            *reinterpret_cast<uint4 *>(vrow + ch * 1024 + p * 16) = make_uint4(0, 0, 0, 0);
                }
            }
            ok = __all_sync(0xFFFFFFFFu, ok && wait_or_abort(&p_empty[u & 1], ((u >> 1) & 1) ^ 1, abort_flag));
            // P^T row: columns 12g..12g+11 = pk, every other column 0
            if (has_row) {
                uint4 q0, q1, q2 = make_uint4(0, 0, 0, 0);
                if (g == 0) {
                    q0 = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    q1 = make_uint4(pk[4], pk[5], 0u, 0u);
                } else {
                    q0 = make_uint4(0, 0, 0, 0);
                    q1 = make_uint4(0u, 0u, pk[0], pk[1]);
                    q2 = make_uint4(pk[2], pk[3], pk[4], pk[5]);
                }
                uint8_t *prw = sP + (u & 1) * P_BYTES + prow;
                *reinterpret_cast<uint4 *>(prw + ((0 ^ pswz) << 4)) = q0;
                *reinterpret_cast<uint4 *>(prw + ((1 ^ pswz) << 4)) = q1;
                *reinterpret_cast<uint4 *>(prw + ((2 ^ pswz) << 4)) = q2;
                *reinterpret_cast<uint4 *>(prw + ((3 ^ pswz) << 4)) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[u & 1]);
        }

        // ------------------------------------------------ output --
        // row sums of each query head: lanes with the same KV head (xor over
        // lane bits 0, 1, 3, 4), then the four warps
#pragma unroll
        for (int n = 0; n < 12; ++n) {
            float vsum = l[n];
            vsum += __shfl_xor_sync(0xFFFFFFFFu, vsum, 1);
            vsum += __shfl_xor_sync(0xFFFFFFFFu, vsum, 2);
            vsum += __shfl_xor_sync(0xFFFFFFFFu, vsum, 8);
            vsum += __shfl_xor_sync(0xFFFFFFFFu, vsum, 16);
            l[n] = vsum;
        }
        if (lane == 0 || lane == 4) {
#pragma unroll
            for (int n = 0; n < 12; ++n) sLsum[(quarter * 2 + g) * 12 + n] = l[n];
        }
        if (nt > 0 && ok && !wait_or_abort(o_full, 0, abort_flag)) ok = false;
        ok = !softmax_bar_or(!ok);  // one decision for the four warps (also orders sLsum)
        const bool have = nt > 0 && ok;
        constexpr float kLn2 = 0.693147180559945309f;
        if (tid < 24) {
            const int gg = tid / 12, nn = tid % 12;
            float lt = sLsum[(0 * 2 + gg) * 12 + nn] + sLsum[(1 * 2 + gg) * 12 + nn] +
                       sLsum[(2 * 2 + gg) * 12 + nn] + sLsum[(3 * 2 + gg) * 12 + nn];
            if (!have) lt = 0.f;
            sInv[tid] = lt > 0.f ? 1.f / lt : 0.f;
            const float lse_v = lt > 0.f ? (sM[tid] + log2f(lt)) * kLn2 : -INFINITY;
            if (!DECODE || a.nsplit == 1) {
                if (a.lse) a.lse[orow_id * kHQ + tid] = lse_v;
            } else {
                a.part_lse[(static_cast<int64_t>(s) * a.nsplit + split) * kHQ + tid] = lse_v;
            }
        }
        named_bar(1, 128);
        __syncwarp();  // the TMEM loads below are warp-collective
        if (have) tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t o[32];
            if (have) {
                tmem_ld32(lane_addr + COL_O + h * NS, o);
                tmem_wait32(o);
            } else {
#pragma unroll
                for (int n = 0; n < 32; ++n) o[n] = 0u;
            }
            const int d = h * 128 + dr;
            if (!DECODE || a.nsplit == 1) {
                uint16_t *orow = a.out + orow_id * (kHQ * kD);
#pragma unroll
                for (int n = 0; n < 24; ++n) {
                    const __nv_bfloat16 y = __float2bfloat16_rn(__uint_as_float(o[n]) * sInv[n]);
                    orow[n * kD + d] = *reinterpret_cast<const uint16_t *>(&y);
                }
            } else {
                float *po = a.part_o + (static_cast<int64_t>(s) * a.nsplit + split) * (kHQ * kD);
#pragma unroll
                for (int n = 0; n < 24; ++n) po[n * kD + d] = __uint_as_float(o[n]) * sInv[n];
            }
        }
        if (!ok && lane == 0) {
            report(a.status, QSA_ERR_TIMEOUT);
            *abort_flag = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == WARP_Q) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace tca

cudaError_t launch_attn_prefill_tc(const AttnArgs &a, const RopeFreqs &f, const CUtensorMap &map_k,
                                   const CUtensorMap &map_v, int64_t key_rows, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(tca::attn_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         tca::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    AttnArgs p = a;
    p.nsplit = 1;
    if (a.L > 0x7FFFFFFF) return cudaErrorInvalidValue;
    tca::attn_tc_kernel<false><<<static_cast<unsigned>(a.L), tca::THREADS, tca::SMEM_BYTES, stream>>>(
        map_k, map_v, p, f, key_rows);
    return cudaGetLastError();
}

cudaError_t launch_attn_decode_tc(const AttnArgs &a, int batch, const RopeFreqs &f, const CUtensorMap &map_k,
                                  const CUtensorMap &map_v, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(tca::attn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         tca::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return launch_pdl(tca::attn_tc_kernel<true>, dim3(a.nsplit, batch), dim3(tca::THREADS),
                      static_cast<size_t>(tca::SMEM_BYTES), stream, map_k, map_v, a, f, a.seq_stride);
}

}  // namespace qsa
