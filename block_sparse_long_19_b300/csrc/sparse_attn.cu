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
//   * one CTA per query (all 24 heads: each gathered row serves both KV heads'
//     12 query heads);
//   * a producer warp issues one 1 KiB cp.async.bulk per key row (both KV
//     heads) into a ring of stages; rows land at a 1040-byte pitch so the
//     tensor-core operand loads (ldmatrix) are free of bank conflicts;
//   * four consumer warps (KV head x stage parity) run QK^T and PV with the
//     warp-level MMA (m16n8k16, bf16 in, fp32 out) and an fp32 online softmax
//     in the log2 domain with a lazy rescale; the two parities merge at the end.
// Decode runs the same kernel over a slice of the selected blocks per CTA
// (split-KV) and a second kernel merges the slices by log-sum-exp.
#include "qsa_common.cuh"
#include "qsa_kernels.h"

namespace qsa {
namespace at {

constexpr int SKEYS = 16;                 // keys per stage = 4 blocks
constexpr int ROWB = kHKV * kD * 2 + 16;  // 1040 B per key row in smem
constexpr int STAGE_BYTES = 2 * SKEYS * ROWB;
constexpr int QROW = kD * 2 + 16;         // 528 B per query row in smem
constexpr int Q_BYTES = kHKV * 16 * QROW;
constexpr int NCONS = 4;
constexpr int THREADS = 32 * (1 + NCONS);
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
static_assert(kHKV * COMB_FLOATS * 4 <= 2 * STAGE_BYTES, "combine buffer must fit in two stages");

__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
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
        qrow = a.q + static_cast<int64_t>(s) * kHQ * kD;
        irow = a.idx + static_cast<int64_t>(s) * a.budget;
        kbase = a.k + static_cast<int64_t>(s) * a.seq_stride * (kHKV * kD);
        vbase = a.v + static_cast<int64_t>(s) * a.seq_stride * (kHKV * kD);
    } else {
        t = a.L - 1 - blockIdx.x;
        qrow = a.q + t * (kHQ * kD);
        irow = a.idx + t * a.budget;
    }
    const int64_t c = t / kBlock;

    // ---------------------------------------------- phase 1: idx, cos/sin --
    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 2);
        }
        fence_barrier_init();
    }
    for (int i = threadIdx.x; i < a.budget; i += THREADS) {
        int b = irow[i];
        if (b < 0 || b > c) b = -1;  // out-of-range entries are ignored
        sIdx[i] = b;
    }
    if (threadIdx.x < 32) {
        float cs, sn;
        rope_cos_sin(t, f.inv_freq[threadIdx.x], cs, sn);
        sCS[threadIdx.x] = cs;
        sCS[32 + threadIdx.x] = sn;
    }
    __syncthreads();

    // ---------------------------------- phase 2: slot count, Q with RoPE --
    if (warp == 0) {
        int last = -1;
        for (int base = 0; base < a.budget; base += 32) {
            const int i = base + lane;
            const bool v = i < a.budget && sIdx[i] >= 0;
            const unsigned ball = __ballot_sync(0xFFFFFFFFu, v);
            if (ball) last = base + 31 - __clz(ball);
        }
        if (lane == 0) sMisc[0] = last + 1;
    }
    for (int i = threadIdx.x; i < kHQ * 32; i += THREADS) {
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
    for (int i = threadIdx.x; i < kHQ * 24; i += THREADS) {
        const int h = i / 24, v = i % 24;
        const uint4 x = *reinterpret_cast<const uint4 *>(qrow + h * kD + kRD + v * 8);
        uint8_t *qr = sQ + (h / kGroup) * 16 * QROW + (h % kGroup) * QROW;
        *reinterpret_cast<uint4 *>(qr + kRD * 2 + v * 16) = x;
    }
    for (int i = threadIdx.x; i < kHKV * 4 * 32; i += THREADS) {  // zero rows 12..15
        const int g = i / 128, r = 12 + (i / 32) % 4, v = i % 32;
        *reinterpret_cast<uint4 *>(sQ + g * 16 * QROW + r * QROW + v * 16) = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();

    const int nslot = sMisc[0];
    const int total_st = (nslot + 3) / 4;
    int st_begin = 0, st_end = total_st;
    if constexpr (DECODE) {
        const int per = (total_st + a.nsplit - 1) / a.nsplit;
        st_begin = split * per;
        st_end = min(total_st, st_begin + per);
        if (st_begin > st_end) st_begin = st_end;
    }

    if (warp == 0) {
        // ------------------------------------------------- producer --
        const int r = lane & 15;
        const int isv = lane >> 4;
        const uint64_t pol = policy_evict_first();
        bool ok = true;
        for (int st = st_begin; st < st_end; ++st) {
            const int local = st - st_begin;
            const int slot = local % NST;
            const uint32_t ph = (local / NST) & 1;
            if (lane == 0) ok = mbar_wait(&empty[slot], ph ^ 1);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], 2 * SKEYS * 1024);
            __syncwarp();
            const int si = st * 4 + (r >> 2);
            const int b = si < a.budget ? sIdx[si] : -1;
            const int64_t j = static_cast<int64_t>(b) * kBlock + (r & 3);
            const bool valid = b >= 0 && j <= t;
            const int64_t row = valid ? j : t;  // masked rows fetch the query's own row
            const uint16_t *src = (isv ? vbase : kbase) + row * (kHKV * kD);
            uint8_t *dst = sSt + slot * STAGE_BYTES + isv * SKEYS * ROWB + r * ROWB;
            bulk_g2s_hint(dst, src, 1024, &full[slot], pol);
        }
        if (!ok && lane == 0) {
            report(a.status, QSA_ERR_TIMEOUT);
            sMisc[1] = 1;
        }
        return;
    }

    // ------------------------------------------------------ consumers --
    const int cw = warp - 1;
    const int g = cw & 1;
    const int par = cw >> 1;
    const int qd = lane & 3;     // column pair within an 8-wide tile
    const int r0 = lane >> 2;    // fragment rows r0 and r0 + 8 (= query heads g*12 + r)
    float O[32][4];
#pragma unroll
    for (int i = 0; i < 32; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY};
    float l_r[2] = {0.f, 0.f};

    const uint32_t q_addr = smem_u32(sQ) + g * 16 * QROW +
                            ((lane & 7) + ((lane >> 3) & 1) * 8) * QROW + (lane >> 4) * 16;
    const int krow_l = (lane & 7) + (lane >> 4) * 8;
    const int kcol_l = ((lane >> 3) & 1) * 16;
    const int vrow_l = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int vcol_l = (lane >> 4) * 16;
    bool ok = true;

    for (int st = st_begin + par; st < st_end; st += 2) {
        const int local = st - st_begin;
        const int slot = local % NST;
        const uint32_t ph = (local / NST) & 1;
        if (!mbar_wait(&full[slot], ph)) { ok = false; break; }
        const uint32_t kb = smem_u32(sSt + slot * STAGE_BYTES) + g * (kD * 2);
        const uint32_t vb = kb + SKEYS * ROWB;

        float S0[4] = {0.f, 0.f, 0.f, 0.f}, S1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
            uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
            ldsm_x4(q_addr + kk * 32, a0, a1, a2, a3);
            ldsm_x4(kb + krow_l * ROWB + kk * 32 + kcol_l, b0, b1, b2, b3);
            mma_bf16_16816(S0, a0, a1, a2, a3, b0, b1);
            mma_bf16_16816(S1, a0, a1, a2, a3, b2, b3);
        }
        // log2-domain logits; mask keys outside the selection or after t
        float z[8] = {S0[0], S0[1], S1[0], S1[1], S0[2], S0[3], S1[2], S1[3]};
        bool need_mask = false;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int si = st * 4 + e;
            const int b = si < a.budget ? sIdx[si] : -1;
            need_mask |= (b < 0) || (b == c);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) z[e] *= a.scale_log2;
        if (need_mask) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int key = (e & 2 ? 8 : 0) + 2 * qd + (e & 1);  // key within the stage
                const int si = st * 4 + (key >> 2);
                const int b = si < a.budget ? sIdx[si] : -1;
                const int64_t j = static_cast<int64_t>(b) * kBlock + (key & 3);
                if (b < 0 || j > t) z[e] = -INFINITY;
            }
        }
        // z[0..3]: row r0 ; z[4..7]: row r0 + 8
        float p[8];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            float mx = fmaxf(fmaxf(z[4 * rr], z[4 * rr + 1]), fmaxf(z[4 * rr + 2], z[4 * rr + 3]));
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
            for (int e = 0; e < 4; ++e) {
                p[4 * rr + e] = dead ? 0.f : exp2f(z[4 * rr + e] - m_r[rr]);
                l_r[rr] += p[4 * rr + e];
            }
        }
        const uint32_t pa0 = pack_bf16(p[0], p[1]);  // row r0,   keys 2qd..   (n-tile 0)
        const uint32_t pa1 = pack_bf16(p[4], p[5]);  // row r0+8, keys 2qd..
        const uint32_t pa2 = pack_bf16(p[2], p[3]);  // row r0,   keys 8+2qd.. (n-tile 1)
        const uint32_t pa3 = pack_bf16(p[6], p[7]);  // row r0+8, keys 8+2qd..
#pragma unroll
        for (int dt = 0; dt < 16; ++dt) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vb + vrow_l * ROWB + dt * 32 + vcol_l, b0, b1, b2, b3);
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

    // ------------------------------------------- merge the two parities --
    named_bar(1, NCONS * 32);  // every consumer is done reading the ring
    float *comb = reinterpret_cast<float *>(sSt) + g * COMB_FLOATS;
    if (par == 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            *reinterpret_cast<float4 *>(&comb[(i * 32 + lane) * 4]) =
                make_float4(O[i][0], O[i][1], O[i][2], O[i][3]);
        *reinterpret_cast<float4 *>(&comb[32 * 32 * 4 + lane * 4]) =
            make_float4(m_r[0], m_r[1], l_r[0], l_r[1]);
    }
    named_bar(1, NCONS * 32);
    if (par == 1) return;
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
        uint16_t *orow = a.out + (DECODE ? static_cast<int64_t>(s) : t) * (kHQ * kD);
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
            float *lrow = a.lse + (DECODE ? static_cast<int64_t>(s) : t) * kHQ;
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

// Merge decode splits: O = sum_i e^(lse_i - M) O_i / sum_i e^(lse_i - M).
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ part_o,
                                                      const float *__restrict__ part_lse,
                                                      int nsplit, uint16_t *__restrict__ out,
                                                      float *__restrict__ lse) {
    const int s = blockIdx.x / kHQ;
    const int h = blockIdx.x % kHQ;
    const int d = threadIdx.x;
    float M = -INFINITY;
    for (int i = 0; i < nsplit; ++i)
        M = fmaxf(M, part_lse[(static_cast<int64_t>(s) * nsplit + i) * kHQ + h]);
    float den = 0.f, acc = 0.f;
    if (M > -INFINITY) {
        for (int i = 0; i < nsplit; ++i) {
            const float li = part_lse[(static_cast<int64_t>(s) * nsplit + i) * kHQ + h];
            if (li == -INFINITY) continue;
            const float wgt = __expf(li - M);
            den += wgt;
            acc += wgt * part_o[((static_cast<int64_t>(s) * nsplit + i) * kHQ + h) * kD + d];
        }
    }
    const float o = den > 0.f ? acc / den : 0.f;
    __nv_bfloat16 ob = __float2bfloat16_rn(o);
    out[(static_cast<int64_t>(s) * kHQ + h) * kD + d] = *reinterpret_cast<uint16_t *>(&ob);
    if (lse && d == 0) lse[static_cast<int64_t>(s) * kHQ + h] = den > 0.f ? M + logf(den) : -INFINITY;
}

}  // namespace at

constexpr int kPrefillStages = 6;
constexpr int kDecodeStages = 3;

cudaError_t launch_attn_prefill(const AttnArgs &a, const RopeFreqs &f, cudaStream_t stream) {
    constexpr int smem = at::smem_bytes<kPrefillStages>();
    cudaError_t e = cudaFuncSetAttribute(at::attn_kernel<kPrefillStages, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    AttnArgs p = a;
    p.nsplit = 1;
    const int64_t grid = a.L;
    if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
    at::attn_kernel<kPrefillStages, false><<<static_cast<unsigned>(grid), at::THREADS, smem, stream>>>(p, f);
    return cudaGetLastError();
}

cudaError_t launch_attn_decode(const AttnArgs &a, int batch, const RopeFreqs &f,
                               cudaStream_t stream) {
    constexpr int smem = at::smem_bytes<kDecodeStages>();
    cudaError_t e = cudaFuncSetAttribute(at::attn_kernel<kDecodeStages, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.nsplit, batch);
    at::attn_kernel<kDecodeStages, true><<<grid, at::THREADS, smem, stream>>>(a, f);
    return cudaGetLastError();
}

cudaError_t launch_attn_combine(const float *part_o, const float *part_lse, int batch,
                                int nsplit, uint16_t *out, float *lse, cudaStream_t stream) {
    at::combine_kernel<<<batch * kHQ, kD, 0, stream>>>(part_o, part_lse, nsplit, out, lse);
    return cudaGetLastError();
}

}  // namespace qsa
