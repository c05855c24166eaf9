// Block-sparse GQA attention over the selected micro-blocks (prefill and the
// split-KV decode step), plus the log-sum-exp combine of decode splits.
//
// What it computes (Qwen3.8-Flash-Next launch post, "Model Architecture /
// Attention: GDN + QSA": attention runs only over the regions the indexer
// selected; model card "Model Overview / Qwen Sparse Attention": 24 query
// heads, 2 KV heads, head dim 256, rotary dim 64): for a query at position t,
// the keys are j with floor(j/4) selected and j <= t; query head h reads KV
// head h/12; O = softmax(Q'K'^T * scale) V with Q' the query after RoPE.
//
// Why this shape: every query gathers its own 2048 keys (4 MiB of K and V
// for both KV heads) and on i.i.d. inputs two queries share almost none of
// them, so the kernel is bound by the gather (about 12 flop per byte), not by
// the tensor cores.  The design therefore spends its effort on the data path:
//   * a query's 24 heads in one CTA (each gathered row serves both KV heads'
//     12 query heads); the prefill kernel (attn_mq_kernel, below) gives a
//     CTA 16 neighbouring queries one after the other with its copy ring
//     running on across them, the decode splits one query's blocks;
//   * two producer warps (one for K, one for V) issue one 4 KiB
//     cp.async.bulk per selected block into a ring of 64 KiB stages of 8
//     blocks; block slots are skewed by 16 bytes so the tensor-core operand
//     loads (ldmatrix) are free of bank conflicts.  4 KiB copies and more
//     than one issuing warp matter: a warp issues a bulk copy only about every
//     100 cycles, so one producer warp could not keep enough bytes in flight;
//   * four consumer warps (KV head x key half of every stage) run QK^T and PV
//     with the warp-level MMA (m16n8k16, bf16 in, fp32 out) and an fp32 online
//     softmax in the log2 domain with a lazy rescale; the two halves merge at
//     the end.  A warp keeps its KV head's query fragments in registers for
//     the whole key loop, so per stage shared memory is read only for K and
//     V.  Every consumer waits on every stage: with an odd ring depth,
//     consumers that skipped stages could wait on a slot two fills ahead,
//     which a one-bit phase parity cannot tell apart.
// Decode runs attn_kernel over a slice of the selected blocks per CTA
// (split-KV) and a second kernel merges the slices by log-sum-exp.
#include "qsa_common.cuh"
#include "qsa_kernels.h"

namespace qsa {
namespace at {

// A stage holds 8 selected blocks (32 keys).  Each block's 4 key rows (both
// KV heads, 1 KiB per row) arrive as one 4 KiB bulk copy into a "slot"; slots
// sit 4096 + 16 bytes apart, so the 8 rows an 8x8 ldmatrix reads (the same
// token of 8 different blocks) fall into 8 different bank groups.
constexpr int SBLK = 8;                   // blocks per stage
constexpr int ROWB = kHKV * kD * 2;       // 1024 B per key row
constexpr int SLOTB = kBlock * ROWB + 16; // 4112 B per block slot
constexpr int KV_BYTES = SBLK * SLOTB;    // K (or V) part of a stage
constexpr int STAGE_BYTES = 2 * KV_BYTES;
constexpr int QROW = kD * 2 + 16;         // 528 B per query row in smem
constexpr int Q_BYTES = kHKV * 16 * QROW;
constexpr int NCONS = 4;
constexpr int WARP_VPROD = 1 + NCONS;    // the V producer (warp 0 produces K)
constexpr int WARP_PF = 2 + NCONS;       // brings the blocks of later stages into L2
constexpr int PF_AHEAD = 10;             // stages the L2 prefetch runs ahead of the K producer
constexpr int THREADS = 32 * (3 + NCONS);
constexpr int OFF_BAR = 0;
constexpr int OFF_IDX = 128;
constexpr int OFF_CS = OFF_IDX + kMaxBudget * 4;
constexpr int OFF_MISC = OFF_CS + 64 * 4;
constexpr int OFF_Q = ((OFF_MISC + 16 + 127) / 128) * 128;
constexpr int OFF_ST = ((OFF_Q + Q_BYTES + 127) / 128) * 128;
template <int NST>
constexpr int smem_bytes() {
    return OFF_ST + NST * STAGE_BYTES;
}
// combine buffer (reuses the stage ring after the main loop): per KV head
// 32 lanes x (32 dim tiles x 4 + 4) floats
constexpr int COMB_FLOATS = 32 * (32 * 4 + 4);
static_assert(kHKV * COMB_FLOATS * 4 <= STAGE_BYTES, "combine buffer must fit in one stage");

__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// named_bar that also returns whether any of the n threads passed pred = true
__device__ __forceinline__ bool named_bar_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

template <int NST, bool DECODE>
__global__ void __launch_bounds__(THREADS, 1) attn_kernel(AttnArgs a, RopeFreqs f) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint64_t *empty = full + NST;
    int32_t *sIdx = reinterpret_cast<int32_t *>(smem + OFF_IDX);
    float *sCS = reinterpret_cast<float *>(smem + OFF_CS);
    volatile int *sMisc = reinterpret_cast<volatile int *>(smem + OFF_MISC);
    uint8_t *sQ = smem + OFF_Q;
    uint8_t *sSt = smem + OFF_ST;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ------------------------------------------------------ work item --
    int64_t t;
    int64_t orow_id;  // output row: the sequence (decode) or the query row (prefill)
    int s = 0, split = 0;
    const uint16_t *qrow;
    const int32_t *irow;
    const uint16_t *kbase = a.k;
    const uint16_t *vbase = a.v;
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
        kbase = a.k + static_cast<int64_t>(s) * a.seq_stride * (kHKV * kD);
        vbase = a.v + static_cast<int64_t>(s) * a.seq_stride * (kHKV * kD);
    } else {
        orow_id = a.L - 1 - blockIdx.x;
        t = a.q_off + orow_id;
        qrow = a.q + orow_id * (kHQ * kD);
        irow = a.idx + orow_id * a.budget;
    }
    const int64_t c = t / kBlock;

    // ---------------------------------------------- phase 1: idx, cos/sin --
    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 2);  // the K and the V producer arrive
            mbar_init(&empty[i], NCONS);
        }
        sMisc[2] = -1;  // the last stage the K producer has issued
        fence_barrier_init();
    }
    if (threadIdx.x < 32) {
        float cs, sn;
        rope_cos_sin(t, f.inv_freq[threadIdx.x], cs, sn);
        sCS[threadIdx.x] = cs;
        sCS[32 + threadIdx.x] = sn;
    }
    auto load_idx = [&]() {
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
    };
    // the consumer warps put Q (with RoPE) into shared memory
    auto q_rope = [&]() {
        const int ct = threadIdx.x - 32;
        constexpr int CT = NCONS * 32;
        for (int i = ct; i < kHQ * 32; i += CT) {
            const int h = i >> 5, r = i & 31;
            const float x1 = __uint_as_float(static_cast<uint32_t>(qrow[h * kD + r]) << 16);
            const float x2 = __uint_as_float(static_cast<uint32_t>(qrow[h * kD + r + 32]) << 16);
            const float cs = sCS[r], sn = sCS[32 + r];
            __nv_bfloat16 y1 = __float2bfloat16_rn(fmaf(x1, cs, -x2 * sn));
            __nv_bfloat16 y2 = __float2bfloat16_rn(fmaf(x2, cs, x1 * sn));
            uint8_t *qr = sQ + (h / kGroup) * 16 * QROW + (h % kGroup) * QROW;
            reinterpret_cast<__nv_bfloat16 *>(qr)[r] = y1;
            reinterpret_cast<__nv_bfloat16 *>(qr)[r + 32] = y2;
        }
        for (int i = ct; i < kHQ * 24; i += CT) {
            const int h = i / 24, v = i % 24;
            const uint4 x = *reinterpret_cast<const uint4 *>(qrow + h * kD + kRD + v * 8);
            uint8_t *qr = sQ + (h / kGroup) * 16 * QROW + (h % kGroup) * QROW;
            *reinterpret_cast<uint4 *>(qr + kRD * 2 + v * 16) = x;
        }
        for (int i = ct; i < kHKV * 4 * 32; i += CT) {  // zero rows 12..15
            const int g = i / 128, r = 12 + (i / 32) % 4, v = i % 32;
            *reinterpret_cast<uint4 *>(sQ + g * 16 * QROW + r * QROW + v * 16) = make_uint4(0, 0, 0, 0);
        }
        named_bar(1, CT);  // Q complete before any consumer reads it
    };
    const bool consumer = warp > 0 && warp <= NCONS;
    if constexpr (DECODE) {
        // the query, its RoPE and the barriers do not depend on the decode
        // indexer: they are set up while it finishes, then the selection is read
        pdl_trigger();
        __syncthreads();
        if (consumer) q_rope();
        pdl_wait();  // the selection of the decode indexer
        load_idx();
        __syncthreads();
    } else {
        load_idx();
        __syncthreads();
    }

    // ---------------------------------- phase 2: slot count, Q with RoPE --
    // Every warp counts the used slots itself; in prefill the producer starts
    // its copies right away while the consumer warps put Q (with RoPE) into
    // shared memory, so the first stages are in flight during that set-up.
    int nslot = 0;
    for (int base = 0; base < a.budget; base += 32) {
        const int i = base + lane;
        const unsigned ball = __ballot_sync(0xFFFFFFFFu, i < a.budget && sIdx[i] >= 0);
        if (ball) nslot = base + 32 - __clz(ball);
    }
    const int total_st = (nslot + SBLK - 1) / SBLK;
    int st_begin = 0, st_end = total_st;
    if constexpr (DECODE) {
        const int per = (total_st + a.nsplit - 1) / a.nsplit;
        st_begin = split * per;
        st_end = min(total_st, st_begin + per);
        if (st_begin > st_end) st_begin = st_end;
    } else {
        if (consumer) q_rope();
    }

    if (warp == WARP_PF) {
        // ------------------------------------------------ L2 prefetch --
        // The ring holds NST stages, about two of them in flight: per SM
        // that is too few bytes to cover the HBM latency at full bandwidth,
        // so the kernel needs many SMs to reach it.  This warp brings the K
        // and V blocks of stages up to PF_AHEAD ahead of the K producer into
        // L2 (lanes 0-7 K, 8-15 V), so the ring's copies are served from L2
        // and fewer SMs saturate HBM.  A hint only: it gives up (nothing else
        // depends on it) if the producer stalls.
        const unsigned long long t0 = globaltimer();
        const int sl = lane & 7;
        const bool isv = lane >= 8;
        for (int st = st_begin + NST; st < st_end; ++st) {
            bool go = true;
            while (sMisc[2] < st - PF_AHEAD) {
                if (sMisc[1] || globaltimer() - t0 > kWaitLimitNs) { go = false; break; }
                __nanosleep(256);
            }
            if (!__all_sync(0xFFFFFFFFu, go)) break;
            if (lane < 16) {
                const int si = st * SBLK + sl;
                const int b = si < a.budget ? sIdx[si] : -1;
                if (b >= 0 && b < c)
                    prefetch_l2_bulk((isv ? vbase : kbase) + static_cast<int64_t>(b) * kBlock * (kHKV * kD),
                                     kBlock * ROWB);
            }
        }
        return;
    }

    if (warp == 0 || warp == WARP_VPROD) {
        // ------------------------------------------------ producers --
        // warp 0 copies K, warp WARP_VPROD copies V: lanes 0..7 the block of
        // slot `lane`.  One warp issues a bulk copy only every ~100 cycles, so
        // two producers keep twice the copies in flight.
        // A past block (b < c, all rows <= t) is one 4 KiB copy.  The current
        // block and padding slots are copied row by row; a row that must not
        // be attended (j > t, or no block) fetches the query's own row t, so
        // every byte read is inside the tensor and finite.
        const int sl = lane & 7;
        const int isv = warp == WARP_VPROD ? 1 : 0;
        const uint64_t pol = policy_evict_first();
        bool ok = true;
        for (int st = st_begin; st < st_end; ++st) {
            const int local = st - st_begin;
            const int slot = local % NST;
            const uint32_t ph = (local / NST) & 1;
            if (lane == 0) ok = mbar_wait(&empty[slot], ph ^ 1);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[slot], SBLK * kBlock * ROWB);  // this producer's half
                if (!isv) sMisc[2] = st;  // paces the L2 prefetch
            }
            __syncwarp();
            if (lane < SBLK) {
                const int si = st * SBLK + sl;
                const int b = si < a.budget ? sIdx[si] : -1;
                const uint16_t *base = isv ? vbase : kbase;
                uint8_t *dst = sSt + slot * STAGE_BYTES + isv * KV_BYTES + sl * SLOTB;
                if (b >= 0 && b < c) {
                    bulk_g2s_hint(dst, base + static_cast<int64_t>(b) * kBlock * (kHKV * kD),
                                  kBlock * ROWB, &full[slot], pol);
                } else {
#pragma unroll
                    for (int r = 0; r < kBlock; ++r) {
                        const int64_t j = static_cast<int64_t>(b) * kBlock + r;
                        const int64_t row = (b >= 0 && j <= t) ? j : t;
                        bulk_g2s_hint(dst + r * ROWB, base + row * (kHKV * kD), ROWB, &full[slot], pol);
                    }
                }
            }
        }
        // the CTA must not finish while its copies can still land: wait for the
        // stages issued last (normal runs find them complete already)
        if (lane == 0) {
            const int first = max(st_begin, st_end - NST);
            for (int st = first; st < st_end; ++st) {
                const int local = st - st_begin;
                if (!mbar_wait(&full[local % NST], (local / NST) & 1)) ok = false;
            }
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok && lane == 0) {
            report(a.status, QSA_ERR_TIMEOUT);
            sMisc[1] = 1;
        }
        return;
    }

    // ------------------------------------------------------ consumers --
    // Every consumer warp takes part in every stage (so no warp can ever wait
    // on a ring slot more than one fill ahead): warp (g, kh) handles KV head g
    // and the key half kh of each stage, i.e. tokens 2kh and 2kh+1 of the 8
    // blocks, and keeps its own online-softmax state; the two key halves are
    // merged at the end.
    const int cw = warp - 1;
    const int g = cw & 1;
    const int kh = cw >> 1;
    const int qd = lane & 3;     // column pair within an 8-wide tile
    const int r0 = lane >> 2;    // fragment rows r0 and r0 + 8 (= query heads g*12 + r)
    float O[32][4];
#pragma unroll
    for (int i = 0; i < 32; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY};
    float l_r[2] = {0.f, 0.f};

    const uint32_t q_addr = smem_u32(sQ) + g * 16 * QROW +
                            ((lane & 7) + ((lane >> 3) & 1) * 8) * QROW + (lane >> 4) * 16;
    // key k of a stage = (token-in-block k / 8, slot k % 8)
    // QK^T B operand (keys x dims): lanes 0-7 / 16-23 -> token 2kh / 2kh+1 of slots 0-7,
    // lanes 8-15 / 24-31 -> dims +8
    const uint32_t k_lane = (lane & 7) * SLOTB + (2 * kh + (lane >> 4)) * ROWB + ((lane >> 3) & 1) * 16;
    // PV B operand via ldmatrix.trans (keys x dims): lanes 0-7 / 8-15 -> token 2kh / 2kh+1
    // of slots 0-7, lanes 16-31 -> dims +8
    const uint32_t v_lane = (lane & 7) * SLOTB + (2 * kh + ((lane >> 3) & 1)) * ROWB + (lane >> 4) * 16;
    bool ok = true;
    // positions fit in 32 bits (at most 2^24 tokens): the key loop runs at
    // the register limit, and 64-bit copies cost it scheduling room
    const int t32 = static_cast<int>(t);
    const int c32 = static_cast<int>(c);
    // the query's A fragments stay in registers for the whole key loop
    uint32_t qf[kD / 16][4];
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) ldsm_x4(q_addr + kk * 32, qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);

    for (int st = st_begin; st < st_end; ++st) {
        const int local = st - st_begin;
        const int slot = local % NST;
        const uint32_t ph = (local / NST) & 1;
        if (!mbar_wait(&full[slot], ph)) { ok = false; break; }
        const uint32_t kb = smem_u32(sSt + slot * STAGE_BYTES) + g * (kD * 2);
        const uint32_t vb = kb + KV_BYTES;

        // S[n][4]: n-tile n = token 2kh + n of the 8 slots
        float S[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n) S[n][0] = S[n][1] = S[n][2] = S[n][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kb + k_lane + kk * 32, b0, b1, b2, b3);
            mma_bf16_16816(S[0], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
            mma_bf16_16816(S[1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
        }
        bool need_mask = false;
#pragma unroll
        for (int e = 0; e < SBLK; ++e) {
            const int si = st * SBLK + e;
            const int b = si < a.budget ? sIdx[si] : -1;
            need_mask |= (b < 0) || (b == c32);
        }
        // S[n][0..1]: row r0, S[n][2..3]: row r0+8; columns = slots 2qd, 2qd+1
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) S[n][e] *= a.scale_log2;
        if (need_mask) {
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int si = st * SBLK + 2 * qd + (e & 1);
                    const int b = si < a.budget ? sIdx[si] : -1;
                    const int j = b * kBlock + 2 * kh + n;
                    if (b < 0 || j > t32) S[n][e] = -INFINITY;
                }
        }
        float pv[2][4];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            float mx = fmaxf(fmaxf(S[0][2 * rr], S[0][2 * rr + 1]), fmaxf(S[1][2 * rr], S[1][2 * rr + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
            if (mx > m_r[rr] + 8.f) {
                const float sc = exp2f(m_r[rr] - mx);
                l_r[rr] *= sc;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    O[i][2 * rr] *= sc;
                    O[i][2 * rr + 1] *= sc;
                }
                m_r[rr] = mx;
            }
            const bool dead = m_r[rr] == -INFINITY;
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float pe = dead ? 0.f : exp2f(S[n][2 * rr + e] - m_r[rr]);
                    pv[n][2 * rr + e] = pe;
                    l_r[rr] += pe;
                }
        }
        // one k-step of 16 keys: token 2kh (n-tile 0) then token 2kh+1 (n-tile 1)
        const uint32_t pa0 = pack_bf16(pv[0][0], pv[0][1]);
        const uint32_t pa1 = pack_bf16(pv[0][2], pv[0][3]);
        const uint32_t pa2 = pack_bf16(pv[1][0], pv[1][1]);
        const uint32_t pa3 = pack_bf16(pv[1][2], pv[1][3]);
        const uint32_t vks = vb + v_lane;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vks + dt * 32, b0, b1, b2, b3);
            mma_bf16_16816(O[2 * dt], pa0, pa1, pa2, pa3, b0, b1);
            mma_bf16_16816(O[2 * dt + 1], pa0, pa1, pa2, pa3, b2, b3);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
    if (!ok) {
        if (lane == 0) {
            report(a.status, QSA_ERR_TIMEOUT);
            sMisc[1] = 1;
        }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        l_r[rr] += __shfl_xor_sync(0xFFFFFFFFu, l_r[rr], 1);
        l_r[rr] += __shfl_xor_sync(0xFFFFFFFFu, l_r[rr], 2);
    }

    // ------------------------------------------ merge the two key halves --
    named_bar(1, NCONS * 32);  // every consumer is done reading the ring
    float *comb = reinterpret_cast<float *>(sSt) + g * COMB_FLOATS;
    if (kh == 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            *reinterpret_cast<float4 *>(&comb[(i * 32 + lane) * 4]) =
                make_float4(O[i][0], O[i][1], O[i][2], O[i][3]);
        *reinterpret_cast<float4 *>(&comb[32 * 32 * 4 + lane * 4]) =
            make_float4(m_r[0], m_r[1], l_r[0], l_r[1]);
    }
    named_bar(1, NCONS * 32);
    if (kh == 1) return;
    const float4 ml = *reinterpret_cast<const float4 *>(&comb[32 * 32 * 4 + lane * 4]);
    const float m1[2] = {ml.x, ml.y}, l1[2] = {ml.z, ml.w};
    float fa[2], fb[2], lt[2], mt[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const float m = fmaxf(m_r[rr], m1[rr]);
        fa[rr] = (m == -INFINITY) ? 0.f : exp2f(m_r[rr] - m);
        fb[rr] = (m == -INFINITY) ? 0.f : exp2f(m1[rr] - m);
        lt[rr] = l_r[rr] * fa[rr] + l1[rr] * fb[rr];
        mt[rr] = m;
    }
    float inv[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) inv[rr] = lt[rr] > 0.f ? 1.f / lt[rr] : 0.f;

    constexpr float kLn2 = 0.693147180559945309f;
    if (!DECODE || a.nsplit == 1) {
        uint16_t *orow = a.out + orow_id * (kHQ * kD);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float4 o1 = *reinterpret_cast<const float4 *>(&comb[(i * 32 + lane) * 4]);
            const float v0 = (O[i][0] * fa[0] + o1.x * fb[0]) * inv[0];
            const float v1 = (O[i][1] * fa[0] + o1.y * fb[0]) * inv[0];
            const float v2 = (O[i][2] * fa[1] + o1.z * fb[1]) * inv[1];
            const float v3 = (O[i][3] * fa[1] + o1.w * fb[1]) * inv[1];
            const int d = i * 8 + 2 * qd;
            if (r0 < kGroup)
                *reinterpret_cast<uint32_t *>(orow + (g * kGroup + r0) * kD + d) = pack_bf16(v0, v1);
            if (r0 + 8 < kGroup)
                *reinterpret_cast<uint32_t *>(orow + (g * kGroup + r0 + 8) * kD + d) = pack_bf16(v2, v3);
        }
        if (a.lse && qd == 0) {
            float *lrow = a.lse + orow_id * kHQ;
            if (r0 < kGroup)
                lrow[g * kGroup + r0] = lt[0] > 0.f ? (mt[0] + log2f(lt[0])) * kLn2 : -INFINITY;
            if (r0 + 8 < kGroup)
                lrow[g * kGroup + r0 + 8] = lt[1] > 0.f ? (mt[1] + log2f(lt[1])) * kLn2 : -INFINITY;
        }
    } else {
        float *po = a.part_o + (static_cast<int64_t>(s) * a.nsplit + split) * (kHQ * kD);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float4 o1 = *reinterpret_cast<const float4 *>(&comb[(i * 32 + lane) * 4]);
            const int d = i * 8 + 2 * qd;
            if (r0 < kGroup)
                *reinterpret_cast<float2 *>(po + (g * kGroup + r0) * kD + d) =
                    make_float2((O[i][0] * fa[0] + o1.x * fb[0]) * inv[0],
                                (O[i][1] * fa[0] + o1.y * fb[0]) * inv[0]);
            if (r0 + 8 < kGroup)
                *reinterpret_cast<float2 *>(po + (g * kGroup + r0 + 8) * kD + d) =
                    make_float2((O[i][2] * fa[1] + o1.z * fb[1]) * inv[1],
                                (O[i][3] * fa[1] + o1.w * fb[1]) * inv[1]);
        }
        if (qd == 0) {
            float *pl = a.part_lse + (static_cast<int64_t>(s) * a.nsplit + split) * kHQ;
            if (r0 < kGroup)
                pl[g * kGroup + r0] = lt[0] > 0.f ? (mt[0] + log2f(lt[0])) * kLn2 : -INFINITY;
            if (r0 + 8 < kGroup)
                pl[g * kGroup + r0 + 8] = lt[1] > 0.f ? (mt[1] + log2f(lt[1])) * kLn2 : -INFINITY;
        }
    }
}

// ---------------------------------------------------------------------------
// Prefill attention, several query rows per CTA.  One query's 64 stages take
// about 80 us of an SM at 1M tokens, and a CTA that handles a single query
// spends several of them on its own start and end (the index row and the
// query are read, the first stage's copies wait for memory, the key halves
// are merged and the output written) while the SM's copies idle.  Here a CTA
// handles up to ROWS rows and its ring of stages runs on across their
// boundaries: the producers start the next row's copies while the consumers
// still work through the last stages of the row before and merge its key
// halves.
// CTA b takes rows b*ROWS .. b*ROWS+ROWS-1 counted from the last one
// (longest first), neighbours, whose selections overlap most: a row's
// blocks are often still in L2 from the row before on the same SM (handing
// out rows one at a time from a counter, so that the SMs worked on
// neighbours at the same time instead, measured slower on topic-segment
// inputs, 1M tokens: 419 vs 403 ms).  CTAs stay short (about 1.2 ms at 1M),
// so SMs come free regularly for work on other streams.
// A loader warp prepares each row in one of two query slots as soon as the
// row two before has been released: the sanitised index row and the row's
// position first (the producers start on those), then Q with RoPE in the
// tensor-core layout (the consumers need that too).
//   warp 0      K producer          warps 1-4  consumers (as in attn_kernel)
//   warp 5      V producer          warp 6     L2 prefetch (a hint)
//   warp 7      loader
// Every role walks the same rows in the same order.  A slot's fills and
// releases alternate (a row's slot is refilled only after every producer
// and consumer lane released it), so no waiter can see a slot two fills
// ahead; the ring stages are numbered across rows and every consumer waits
// on every stage, as in attn_kernel.
constexpr int MQ_NQ = 2;                                  // query slots
constexpr int MQ_THREADS = 32 * 8;
constexpr int MQ_WARP_VPROD = 5, MQ_WARP_PF = 6, MQ_WARP_LOAD = 7;
constexpr int MQ_QSLOT = kHKV * kGroup * QROW;            // 12 live rows per KV head
constexpr int MQ_OFF_BAR = 0;                              // full, empty, qidx, qrdy, qempty
constexpr int MQ_OFF_MISC = 128;                           // [1] abort, [2] last K stage issued
constexpr int MQ_OFF_QINFO = 192;                          // per slot {t, output row, used slots}
constexpr int MQ_OFF_IDX = 256;
constexpr int MQ_OFF_ZERO = MQ_OFF_IDX + MQ_NQ * kMaxBudget * 4;  // one zero query row
constexpr int MQ_OFF_Q = ((MQ_OFF_ZERO + QROW + 127) / 128) * 128;
constexpr int MQ_OFF_ST = ((MQ_OFF_Q + MQ_NQ * MQ_QSLOT + 127) / 128) * 128;
constexpr int MQ_QE_COUNT = 2 * 32 + NCONS * 32;          // lanes that release a slot
constexpr int MQ_COMB_TILES = 8;                           // O tiles merged per round
#ifndef QSA_ATTN_MQ_PF_AHEAD
#define QSA_ATTN_MQ_PF_AHEAD 2
#endif
// Stages the L2 prefetch runs ahead of the K producer.  With the ring
// running on across rows the prefetch never pauses, and a longer lead keeps
// so much of every SM's future data in L2 that it evicts itself (1M tokens,
// 4 rows per CTA: 2 stages 539 ms, 4 stages 544, 8 stages 588).
constexpr int MQ_PF_AHEAD = QSA_ATTN_MQ_PF_AHEAD;
constexpr unsigned MQ_LOADER_SLEEP_NS = 1000;
template <int NST>
constexpr int mq_smem_bytes() {
    return MQ_OFF_ST + NST * STAGE_BYTES;
}
static_assert(kHKV * (MQ_COMB_TILES * 32 * 4 + 32 * 4) * 4 <= MQ_QSLOT, "merge buffer must fit in a query slot");
static_assert(mq_smem_bytes<3>() <= 227 * 1024, "shared memory");

struct MqInfo {
    int64_t t;
    int64_t orow;
    int nslot;  // used index slots
    int pad;
};

template <int NST, int ROWS>
__global__ void __launch_bounds__(MQ_THREADS, 1) attn_mq_kernel(AttnArgs a, RopeFreqs f) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + MQ_OFF_BAR);
    uint64_t *empty = full + NST;
    uint64_t *qidx = empty + NST;   // a slot's index row and position are in place
    uint64_t *qrdy = qidx + MQ_NQ;  // ... and its Q with RoPE as well
    uint64_t *qempty = qrdy + MQ_NQ;
    volatile int *sMisc = reinterpret_cast<volatile int *>(smem + MQ_OFF_MISC);
    MqInfo *sInfo = reinterpret_cast<MqInfo *>(smem + MQ_OFF_QINFO);
    int32_t *sIdxAll = reinterpret_cast<int32_t *>(smem + MQ_OFF_IDX);
    uint8_t *sZero = smem + MQ_OFF_ZERO;
    uint8_t *sQAll = smem + MQ_OFF_Q;
    uint8_t *sSt = smem + MQ_OFF_ST;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * ROWS;
    const int nq = static_cast<int>(a.L - row0 < ROWS ? a.L - row0 : ROWS);  // rows of this CTA
    const uint16_t *kbase = a.k;
    const uint16_t *vbase = a.v;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 2);  // the K and the V producer arrive
            mbar_init(&empty[i], NCONS);
        }
        for (int i = 0; i < MQ_NQ; ++i) {
            mbar_init(&qidx[i], 32);  // every loader lane
            mbar_init(&qrdy[i], 32);
            mbar_init(&qempty[i], MQ_QE_COUNT);
        }
        sMisc[1] = 0;
        sMisc[2] = -1;
        fence_barrier_init();
    }
    __syncthreads();

    // a bounded wait that also gives up once another role has failed
    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity)) return true;
        const unsigned long long t0 = globaltimer();
        while (true) {
#pragma unroll 1
            for (int i = 0; i < 32; ++i)
                if (mbar_try_wait(bar, parity)) return true;
            if (sMisc[1] || globaltimer() - t0 > kWaitLimitNs) return false;
        }
    };
    // the loader's wait for a slot lasts about a row: it polls with pauses,
    // so that it takes no issue slots from the consumer warp it shares a
    // scheduler with
    auto wait_slow = [&](uint64_t *bar, uint32_t parity) -> bool {
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(bar, parity)) {
            if (sMisc[1] || globaltimer() - t0 > kWaitLimitNs) return false;
            __nanosleep(MQ_LOADER_SLEEP_NS);
        }
        return true;
    };
    auto fail = [&]() {
        if (lane == 0) {
            report(a.status, QSA_ERR_TIMEOUT);
            sMisc[1] = 1;
        }
    };

    if (warp == MQ_WARP_LOAD) {
        // ------------------------------------------------------ loader --
#pragma unroll 1
        for (int j = 0; j < nq; ++j) {
            const int q = j % MQ_NQ;
            if (!__all_sync(0xFFFFFFFFu, wait_slow(&qempty[q], ((j / MQ_NQ) & 1) ^ 1))) {
                fail();
                break;
            }
            const int64_t orow = a.L - 1 - (row0 + j);  // longest first
            const int64_t t = a.q_off + orow;
            const int64_t c = t / kBlock;
            const int32_t *irow = a.idx + orow * a.budget;
            int32_t *sIdx = sIdxAll + q * kMaxBudget;
            int nslot = 0;
#pragma unroll 4
            for (int base = 0; base < a.budget; base += 32) {
                const int i = base + lane;
                int b = i < a.budget ? irow[i] : -1;
#if QSA_DEBUG_CHECKS
                if (i < a.budget) {
                    const int nxt = i + 1 < a.budget ? irow[i + 1] : -1;
                    bool row_ok = b >= -1 && b <= c && (i > 0 || b >= 0);
                    if (b >= 0) row_ok = row_ok && (nxt < 0 ? b == c : b < nxt);
                    else row_ok = row_ok && nxt < 0;
                    debug_check(a.status, row_ok);
                }
#endif
                if (b < 0 || b > c) b = -1;  // out-of-range entries are ignored
                if (i < a.budget) sIdx[i] = b;
                const unsigned ball = __ballot_sync(0xFFFFFFFFu, b >= 0);
                if (ball) nslot = base + 32 - __clz(ball);
            }
            if (lane == 0) {
                sInfo[q].t = t;
                sInfo[q].orow = orow;
                sInfo[q].nslot = nslot;
            }
            __syncwarp();
            mbar_arrive(&qidx[q]);  // the producers can start on this row
            // Q with RoPE: lane r rotates pair (r, r + 32) of every head; all
            // of the row's loads are issued before any is used
            const uint16_t *qrow = a.q + orow * (kHQ * kD);
            uint8_t *sQ = sQAll + q * MQ_QSLOT;
            uint16_t x1[kHQ], x2[kHQ];
            uint4 xr[kHQ * 24 / 32];
#pragma unroll
            for (int h = 0; h < kHQ; ++h) {
                x1[h] = qrow[h * kD + lane];
                x2[h] = qrow[h * kD + lane + 32];
            }
#pragma unroll
            for (int u = 0; u < kHQ * 24 / 32; ++u) {
                const int i = u * 32 + lane, h = i / 24, v = i % 24;
                xr[u] = *reinterpret_cast<const uint4 *>(qrow + h * kD + kRD + v * 8);
            }
            float cs, sn;
            rope_cos_sin(t, f.inv_freq[lane], cs, sn);
#pragma unroll
            for (int h = 0; h < kHQ; ++h) {
                const float y1 = __uint_as_float(static_cast<uint32_t>(x1[h]) << 16);
                const float y2 = __uint_as_float(static_cast<uint32_t>(x2[h]) << 16);
                uint8_t *qr = sQ + (h / kGroup) * kGroup * QROW + (h % kGroup) * QROW;
                reinterpret_cast<__nv_bfloat16 *>(qr)[lane] = __float2bfloat16_rn(fmaf(y1, cs, -y2 * sn));
                reinterpret_cast<__nv_bfloat16 *>(qr)[lane + 32] = __float2bfloat16_rn(fmaf(y2, cs, y1 * sn));
            }
#pragma unroll
            for (int u = 0; u < kHQ * 24 / 32; ++u) {
                const int i = u * 32 + lane, h = i / 24, v = i % 24;
                uint8_t *qr = sQ + (h / kGroup) * kGroup * QROW + (h % kGroup) * QROW;
                *reinterpret_cast<uint4 *>(qr + kRD * 2 + v * 16) = xr[u];
            }
            if (j == 0)
                for (int i = lane; i < QROW / 16; i += 32)
                    *reinterpret_cast<uint4 *>(sZero + i * 16) = make_uint4(0, 0, 0, 0);
            __syncwarp();
            mbar_arrive(&qrdy[q]);
        }
    } else if (warp == MQ_WARP_PF) {
        // ------------------------------------------------ L2 prefetch --
        // As in attn_kernel: the K and V blocks of the stages up to
        // MQ_PF_AHEAD ahead of the K producer, across row boundaries.  A
        // hint only: it stops at once if anything looks wrong (a failure, a
        // time limit, or the producers already past the row it waits for).
        const unsigned long long t0 = globaltimer();
        const int sl = lane & 7;
        const bool isv = lane >= 8;
        int gbase = 0;  // ring stage number of the row's first stage
        bool go = true;
#pragma unroll 1
        for (int j = 0; j < nq && go; ++j) {
            const int q = j % MQ_NQ;
            while (!mbar_try_wait(&qidx[q], (j / MQ_NQ) & 1)) {
                if (sMisc[1] || globaltimer() - t0 > kWaitLimitNs) { go = false; break; }
                if (sMisc[2] >= gbase) {  // the producers are into this row: ready, or this warp is behind
                    go = mbar_try_wait(&qidx[q], (j / MQ_NQ) & 1);
                    break;
                }
                __nanosleep(256);
            }
            go = __all_sync(0xFFFFFFFFu, go);
            if (!go) break;
            const int64_t c = sInfo[q].t / kBlock;
            const int total_st = (sInfo[q].nslot + SBLK - 1) / SBLK;
            const int32_t *sIdx = sIdxAll + q * kMaxBudget;
#pragma unroll 1
            for (int st = 0; st < total_st && go; ++st) {
                const int gs = gbase + st;
                if (gs < NST) continue;  // the producers issue these at once
                int kst;
                while ((kst = sMisc[2]) < gs - MQ_PF_AHEAD) {
                    if (sMisc[1] || globaltimer() - t0 > kWaitLimitNs) { go = false; break; }
                    __nanosleep(256);
                }
                go = __all_sync(0xFFFFFFFFu, go);
                if (!go || __shfl_sync(0xFFFFFFFFu, kst, 0) >= gs) continue;  // stopped, or already issued
                if (lane < 16) {
                    const int si = st * SBLK + sl;
                    const int b = si < a.budget ? sIdx[si] : -1;
                    if (b >= 0 && b < c)
                        prefetch_l2_bulk((isv ? vbase : kbase) + static_cast<int64_t>(b) * kBlock * (kHKV * kD),
                                         kBlock * ROWB);
                }
            }
            gbase += total_st;
        }
    } else if (warp == 0 || warp == MQ_WARP_VPROD) {
        // ------------------------------------------------ producers --
        // As in attn_kernel, with the ring's stage number running on
        // across the rows.
        const int sl = lane & 7;
        const int isv = warp == MQ_WARP_VPROD ? 1 : 0;
        const uint64_t pol = policy_evict_first();
        bool ok = true;
        int g = 0;  // ring stage number
#pragma unroll 1
        for (int j = 0; j < nq; ++j) {
            const int q = j % MQ_NQ;
            ok = __all_sync(0xFFFFFFFFu, wait(&qidx[q], (j / MQ_NQ) & 1));
            if (!ok) break;
            const int64_t t = sInfo[q].t;
            const int64_t c = t / kBlock;
            const int total_st = (sInfo[q].nslot + SBLK - 1) / SBLK;
            const int32_t *sIdx = sIdxAll + q * kMaxBudget;
#pragma unroll 1
            for (int st = 0; st < total_st; ++st, ++g) {
                const int slot = g % NST;
                const uint32_t ph = (g / NST) & 1;
                if (lane == 0) ok = wait(&empty[slot], ph ^ 1);
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                if (!ok) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[slot], SBLK * kBlock * ROWB);  // this producer's half
                    if (!isv) sMisc[2] = g;  // paces the L2 prefetch
                }
                __syncwarp();
                if (lane < SBLK) {
                    const int si = st * SBLK + sl;
                    const int b = si < a.budget ? sIdx[si] : -1;
                    const uint16_t *base = isv ? vbase : kbase;
                    uint8_t *dst = sSt + slot * STAGE_BYTES + isv * KV_BYTES + sl * SLOTB;
                    if (b >= 0 && b < c) {
                        bulk_g2s_hint(dst, base + static_cast<int64_t>(b) * kBlock * (kHKV * kD),
                                      kBlock * ROWB, &full[slot], pol);
                    } else {
#pragma unroll
                        for (int r = 0; r < kBlock; ++r) {
                            const int64_t jj = static_cast<int64_t>(b) * kBlock + r;
                            const int64_t row = (b >= 0 && jj <= t) ? jj : t;
                            bulk_g2s_hint(dst + r * ROWB, base + row * (kHKV * kD), ROWB, &full[slot], pol);
                        }
                    }
                }
            }
            if (!ok) break;
            __syncwarp();
            mbar_arrive(&qempty[q]);  // this row's indices are no longer read here
        }
        // the CTA must not finish while its copies can still land
        if (lane == 0) {
            for (int gg = max(0, g - NST); gg < g; ++gg)
                if (!mbar_wait(&full[gg % NST], (gg / NST) & 1)) ok = false;
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) fail();
    } else {
        // -------------------------------------------------- consumers --
        // The stage arithmetic of attn_kernel; between rows the two key
        // halves are merged through the finished row's query slot (its Q is
        // in registers by then), eight O tiles at a time.  A failed wait
        // sets the abort flag and skips the rest of the row's work, but the
        // warp still passes the row's named barriers, and the four consumer
        // warps decide together (a barrier reduction) whether to go on, so
        // none is ever left at a barrier that the others no longer reach.
        const int cw = warp - 1;
        const int g = cw & 1;
        const int kh = cw >> 1;
        const int qd = lane & 3;
        const int r0 = lane >> 2;
        const int qrow_lane = (lane & 7) + ((lane >> 3) & 1) * 8;  // fragment row this lane addresses
        const uint32_t k_lane = (lane & 7) * SLOTB + (2 * kh + (lane >> 4)) * ROWB + ((lane >> 3) & 1) * 16;
        const uint32_t v_lane = (lane & 7) * SLOTB + (2 * kh + ((lane >> 3) & 1)) * ROWB + (lane >> 4) * 16;
        constexpr float kLn2 = 0.693147180559945309f;
        bool ok = true;
        int gs = 0;  // ring stage number
#pragma unroll 1
        for (int j = 0; j < nq; ++j) {
            const int q = j % MQ_NQ;
            ok = __all_sync(0xFFFFFFFFu, wait(&qrdy[q], (j / MQ_NQ) & 1));  // also covers the index row
            if (!ok) fail();
            // a failed wait: the four warps agree before any of them leaves
            if (named_bar_or(1, NCONS * 32, !ok)) break;
            // positions fit in 32 bits (at most 2^24 tokens); the stage loop
            // runs at the register limit, so it keeps as little as it can
            const int t = static_cast<int>(sInfo[q].t);
            const int c = t / kBlock;
            const int total_st = (sInfo[q].nslot + SBLK - 1) / SBLK;
            const int32_t *sIdx = sIdxAll + q * kMaxBudget;
            uint8_t *sQ = sQAll + q * MQ_QSLOT;
            // rows 12..15 of the A fragments are zero (12 query heads per KV head)
            const uint32_t q_addr = qrow_lane < kGroup
                                        ? smem_u32(sQ) + g * kGroup * QROW + qrow_lane * QROW + (lane >> 4) * 16
                                        : smem_u32(sZero) + (lane >> 4) * 16;
            uint32_t qf[kD / 16][4];
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
                ldsm_x4(q_addr + kk * 32, qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
            float O[32][4];
#pragma unroll
            for (int i = 0; i < 32; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;
            float m_r[2] = {-INFINITY, -INFINITY};
            float l_r[2] = {0.f, 0.f};

#pragma unroll 1
            for (int st = 0; st < total_st; ++st, ++gs) {
                const int slot = gs % NST;
                const uint32_t ph = (gs / NST) & 1;
                if (!__all_sync(0xFFFFFFFFu, wait(&full[slot], ph))) {
                    ok = false;
                    fail();
                    break;
                }
                const uint32_t kb = smem_u32(sSt + slot * STAGE_BYTES) + g * (kD * 2);
                const uint32_t vb = kb + KV_BYTES;
                float S[2][4];
#pragma unroll
                for (int n = 0; n < 2; ++n) S[n][0] = S[n][1] = S[n][2] = S[n][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kb + k_lane + kk * 32, b0, b1, b2, b3);
                    mma_bf16_16816(S[0], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
                    mma_bf16_16816(S[1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
                }
                bool need_mask = false;
#pragma unroll
                for (int e = 0; e < SBLK; ++e) {
                    const int si = st * SBLK + e;
                    const int b = si < a.budget ? sIdx[si] : -1;
                    need_mask |= (b < 0) || (b == c);
                }
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) S[n][e] *= a.scale_log2;
                if (need_mask) {
#pragma unroll
                    for (int n = 0; n < 2; ++n)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int si = st * SBLK + 2 * qd + (e & 1);
                            const int b = si < a.budget ? sIdx[si] : -1;
                            const int jj = b * kBlock + 2 * kh + n;
                            if (b < 0 || jj > t) S[n][e] = -INFINITY;
                        }
                }
                float pv[2][4];
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    float mx = fmaxf(fmaxf(S[0][2 * rr], S[0][2 * rr + 1]), fmaxf(S[1][2 * rr], S[1][2 * rr + 1]));
                    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
                    if (mx > m_r[rr] + 8.f) {
                        const float sc = exp2f(m_r[rr] - mx);
                        l_r[rr] *= sc;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            O[i][2 * rr] *= sc;
                            O[i][2 * rr + 1] *= sc;
                        }
                        m_r[rr] = mx;
                    }
                    const bool dead = m_r[rr] == -INFINITY;
#pragma unroll
                    for (int n = 0; n < 2; ++n)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float pe = dead ? 0.f : exp2f(S[n][2 * rr + e] - m_r[rr]);
                            pv[n][2 * rr + e] = pe;
                            l_r[rr] += pe;
                        }
                }
                const uint32_t pa0 = pack_bf16(pv[0][0], pv[0][1]);
                const uint32_t pa1 = pack_bf16(pv[0][2], pv[0][3]);
                const uint32_t pa2 = pack_bf16(pv[1][0], pv[1][1]);
                const uint32_t pa3 = pack_bf16(pv[1][2], pv[1][3]);
                const uint32_t vks = vb + v_lane;
#pragma unroll
                for (int dt = 0; dt < 16; ++dt) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(vks + dt * 32, b0, b1, b2, b3);
                    mma_bf16_16816(O[2 * dt], pa0, pa1, pa2, pa3, b0, b1);
                    mma_bf16_16816(O[2 * dt + 1], pa0, pa1, pa2, pa3, b2, b3);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                l_r[rr] += __shfl_xor_sync(0xFFFFFFFFu, l_r[rr], 1);
                l_r[rr] += __shfl_xor_sync(0xFFFFFFFFu, l_r[rr], 2);
            }

            // ------------------------------ merge the two key halves --
            float *comb = reinterpret_cast<float *>(sQ) + g * (MQ_COMB_TILES * 32 * 4 + 32 * 4);
            float *ml_buf = comb + MQ_COMB_TILES * 32 * 4;
            named_bar(1, NCONS * 32);  // every consumer has its Q fragments and is past the ring
            if (kh == 1)
                *reinterpret_cast<float4 *>(&ml_buf[lane * 4]) = make_float4(m_r[0], m_r[1], l_r[0], l_r[1]);
            float fa[2] = {0.f, 0.f}, fb[2] = {0.f, 0.f}, lt[2] = {0.f, 0.f}, mt[2] = {0.f, 0.f},
                  inv[2] = {0.f, 0.f};
            const int64_t orow_id = *reinterpret_cast<volatile int64_t *>(&sInfo[q].orow);
            uint16_t *orow = a.out + orow_id * (kHQ * kD);
            bool stop = false;
#pragma unroll
            for (int rd = 0; rd < 32 / MQ_COMB_TILES; ++rd) {
                if (kh == 1) {
#pragma unroll
                    for (int i = 0; i < MQ_COMB_TILES; ++i) {
                        const int ti = rd * MQ_COMB_TILES + i;
                        *reinterpret_cast<float4 *>(&comb[(i * 32 + lane) * 4]) =
                            make_float4(O[ti][0], O[ti][1], O[ti][2], O[ti][3]);
                    }
                }
                named_bar(1, NCONS * 32);
                if (kh == 0) {
                    if (rd == 0) {
                        const float4 ml = *reinterpret_cast<const float4 *>(&ml_buf[lane * 4]);
                        const float m1[2] = {ml.x, ml.y}, l1[2] = {ml.z, ml.w};
#pragma unroll
                        for (int rr = 0; rr < 2; ++rr) {
                            const float m = fmaxf(m_r[rr], m1[rr]);
                            fa[rr] = (m == -INFINITY) ? 0.f : exp2f(m_r[rr] - m);
                            fb[rr] = (m == -INFINITY) ? 0.f : exp2f(m1[rr] - m);
                            lt[rr] = l_r[rr] * fa[rr] + l1[rr] * fb[rr];
                            mt[rr] = m;
                            inv[rr] = lt[rr] > 0.f ? 1.f / lt[rr] : 0.f;
                        }
                    }
#pragma unroll
                    for (int i = 0; i < MQ_COMB_TILES; ++i) {
                        const int ti = rd * MQ_COMB_TILES + i;
                        const float4 o1 = *reinterpret_cast<const float4 *>(&comb[(i * 32 + lane) * 4]);
                        const float v0 = (O[ti][0] * fa[0] + o1.x * fb[0]) * inv[0];
                        const float v1 = (O[ti][1] * fa[0] + o1.y * fb[0]) * inv[0];
                        const float v2 = (O[ti][2] * fa[1] + o1.z * fb[1]) * inv[1];
                        const float v3 = (O[ti][3] * fa[1] + o1.w * fb[1]) * inv[1];
                        const int d = ti * 8 + 2 * qd;
                        if (ok && r0 < kGroup)
                            *reinterpret_cast<uint32_t *>(orow + (g * kGroup + r0) * kD + d) = pack_bf16(v0, v1);
                        if (ok && r0 + 8 < kGroup)
                            *reinterpret_cast<uint32_t *>(orow + (g * kGroup + r0 + 8) * kD + d) =
                                pack_bf16(v2, v3);
                    }
                }
                if (rd + 1 < 32 / MQ_COMB_TILES) named_bar(1, NCONS * 32);
                else stop = named_bar_or(1, NCONS * 32, !ok || sMisc[1] != 0);
            }
            if (ok && kh == 0 && a.lse && qd == 0) {
                float *lrow = a.lse + orow_id * kHQ;
                if (r0 < kGroup) lrow[g * kGroup + r0] = lt[0] > 0.f ? (mt[0] + log2f(lt[0])) * kLn2 : -INFINITY;
                if (r0 + 8 < kGroup)
                    lrow[g * kGroup + r0 + 8] = lt[1] > 0.f ? (mt[1] + log2f(lt[1])) * kLn2 : -INFINITY;
            }
            if (stop) break;
            mbar_arrive(&qempty[q]);  // the slot's indices, Q and merge buffer are free
        }
    }
}

// Merge decode splits: O = sum_i e^(lse_i - M) O_i / sum_i e^(lse_i - M).
// All of a thread's loads are issued before their values are used (split
// LSEs, then the partial outputs), so the merge costs two round trips to L2
// instead of one per split.
constexpr int kMaxSplits = 16;
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ part_o,
                                                      const float *__restrict__ part_lse,
                                                      int nsplit, uint16_t *__restrict__ out,
                                                      float *__restrict__ lse) {
    pdl_wait();  // the splits' partial outputs
    const int s = blockIdx.x / kHQ;
    const int h = blockIdx.x % kHQ;
    const int d = threadIdx.x;
    float li[kMaxSplits], oi[kMaxSplits];
#pragma unroll
    for (int i = 0; i < kMaxSplits; ++i)
        li[i] = i < nsplit ? __ldcg(part_lse + (static_cast<int64_t>(s) * nsplit + i) * kHQ + h) : -INFINITY;
#pragma unroll
    for (int i = 0; i < kMaxSplits; ++i)
        oi[i] = i < nsplit ? __ldcg(part_o + ((static_cast<int64_t>(s) * nsplit + i) * kHQ + h) * kD + d) : 0.f;
    float M = -INFINITY;
#pragma unroll
    for (int i = 0; i < kMaxSplits; ++i) M = fmaxf(M, li[i]);
    float den = 0.f, acc = 0.f;
    if (M > -INFINITY) {
#pragma unroll
        for (int i = 0; i < kMaxSplits; ++i) {
            if (li[i] == -INFINITY) continue;  // an empty split (or one past nsplit)
            const float wgt = __expf(li[i] - M);
            den += wgt;
            acc += wgt * oi[i];
        }
    }
    const float o = den > 0.f ? acc / den : 0.f;
    __nv_bfloat16 ob = __float2bfloat16_rn(o);
    out[(static_cast<int64_t>(s) * kHQ + h) * kD + d] = *reinterpret_cast<uint16_t *>(&ob);
    if (lse && d == 0) lse[static_cast<int64_t>(s) * kHQ + h] = den > 0.f ? M + logf(den) : -INFINITY;
}

}  // namespace at

constexpr int kPrefillStages = 3;
constexpr int kDecodeStages = 3;

// Query rows per prefill CTA at most (1: attn_kernel, one row per CTA).
#ifndef QSA_ATTN_ROWS_PER_CTA
#define QSA_ATTN_ROWS_PER_CTA 16
#endif
constexpr int kPrefillRows = QSA_ATTN_ROWS_PER_CTA;

cudaError_t launch_attn_prefill(const AttnArgs &a, const RopeFreqs &f, cudaStream_t stream) {
    if (a.L <= 0) return cudaSuccess;
    AttnArgs p = a;
    p.nsplit = 1;
    if constexpr (kPrefillRows > 1) {
        constexpr int smem = at::mq_smem_bytes<kPrefillStages>();
        auto kern = at::attn_mq_kernel<kPrefillStages, kPrefillRows>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        const int64_t grid = (a.L + kPrefillRows - 1) / kPrefillRows;
        if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
        kern<<<static_cast<unsigned>(grid), at::MQ_THREADS, smem, stream>>>(p, f);
        return cudaGetLastError();
    } else {
        constexpr int smem = at::smem_bytes<kPrefillStages>();
        cudaError_t e = cudaFuncSetAttribute(at::attn_kernel<kPrefillStages, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        const int64_t grid = a.L;
        if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
        at::attn_kernel<kPrefillStages, false><<<static_cast<unsigned>(grid), at::THREADS, smem, stream>>>(p, f);
        return cudaGetLastError();
    }
}

cudaError_t launch_attn_decode(const AttnArgs &a, int batch, const RopeFreqs &f,
                               cudaStream_t stream) {
    constexpr int smem = at::smem_bytes<kDecodeStages>();
    cudaError_t e = cudaFuncSetAttribute(at::attn_kernel<kDecodeStages, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(at::attn_kernel<kDecodeStages, true>, dim3(a.nsplit, batch), dim3(at::THREADS),
                      static_cast<size_t>(smem), stream, a, f);
}

cudaError_t launch_attn_combine(const float *part_o, const float *part_lse, int batch,
                                int nsplit, uint16_t *out, float *lse, cudaStream_t stream) {
    return launch_pdl(at::combine_kernel, dim3(batch * kHQ), dim3(kD), 0, stream, part_o, part_lse, nsplit, out,
                      lse);
}

}  // namespace qsa
