// K-prep: micro-block keys of the indexer and RoPE of the attention keys.
//
// Block keys: the launch post of Qwen3.8-Flash-Next ("Model Architecture /
// Attention: GDN + QSA") says the indexer first aggregates the sequence into
// micro-blocks; here a block key is the mean of its 4 indexer keys, summed in
// fp64 in token order, scaled by 1/4 and rounded once to bf16 (nearest-even),
// which is what the indexer's tensor cores then read.
// RoPE: model card "Processing Ultra-Long Texts" (rope_theta, partial rotary
// factor 0.25 -> first 64 of 256 dims), rotate-half pairing (i, i + 32).
//
// Both kernels are HBM-streaming elementwise passes (16-byte vector loads and
// stores, grid-stride over the rows).
#include "qsa_common.cuh"
#include "qsa_kernels.h"

namespace qsa {

// Round a double to bf16, nearest-even, straight from the double's bits:
// keep the top 8 significant bits, decide with the 45 bits below them.
__device__ __forceinline__ uint16_t f64_to_bf16_rne(double x) {
    unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(x));
    const unsigned long long sign = u >> 63;
    const int e = static_cast<int>((u >> 52) & 0x7FF);
    unsigned long long mant = u & 0xFFFFFFFFFFFFFull;
    if (e == 0x7FF) return mant ? 0x7FC0 : static_cast<uint16_t>((sign << 15) | 0x7F80);
    if (e == 0) return static_cast<uint16_t>(sign << 15);  // fp64 subnormal: below bf16 range
    const int ef = e - 1023 + 127;                           // bf16 biased exponent
    unsigned long long sig = mant | (1ull << 52);            // 53-bit significand
    int shift;                                               // bits dropped from sig
    int eo;
    if (ef >= 1) {
        shift = 45;  // keep 8 bits
        eo = ef;
    } else {
        shift = 45 + (1 - ef);  // bf16 subnormal: fewer kept bits
        eo = 0;
        if (shift > 60) return static_cast<uint16_t>(sign << 15);
    }
    unsigned long long keep = sig >> shift;
    const unsigned long long rem = sig & ((1ull << shift) - 1);
    const unsigned long long half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (keep & 1))) keep += 1;
    uint32_t out;
    if (eo >= 1) {
        // keep in [2^7, 2^8]; carry to 2^8 bumps the exponent
        if (keep >> 8) { keep >>= 1; eo += 1; }
        if (eo >= 0xFF) return static_cast<uint16_t>((sign << 15) | 0x7F80);
        out = (static_cast<uint32_t>(eo) << 7) | static_cast<uint32_t>(keep & 0x7F);
    } else {
        // subnormal: keep < 2^7, or == 2^7 which is the smallest normal
        out = static_cast<uint32_t>(keep);
    }
    return static_cast<uint16_t>((sign << 15) | out);
}

__device__ __forceinline__ double bf16_to_f64(uint16_t b) {
    return static_cast<double>(__uint_as_float(static_cast<uint32_t>(b) << 16));
}

// One thread per (sequence, block, 8-dim chunk).
__global__ void __launch_bounds__(256) kprep_blocks_kernel(const uint16_t *__restrict__ ki,
                                                           uint16_t *__restrict__ kblk, int batch,
                                                           int64_t b_lo, int64_t nb, int64_t max_ctx) {
    const int64_t per_seq = (nb - b_lo) * (kDI / 8);
    const int64_t total = per_seq * batch;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t s = i / per_seq;
        const int64_t r = i - s * per_seq;
        const int64_t b = b_lo + r / (kDI / 8);
        const int d8 = static_cast<int>(r % (kDI / 8));
        const uint16_t *src = ki + (s * max_ctx + b * kBlock) * kDI + d8 * 8;
        uint4 v[kBlock];
#pragma unroll
        for (int t = 0; t < kBlock; ++t) v[t] = *reinterpret_cast<const uint4 *>(src + t * kDI);
        uint16_t out[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            double sum = 0.0;
#pragma unroll
            for (int t = 0; t < kBlock; ++t) {
                const uint16_t *h = reinterpret_cast<const uint16_t *>(&v[t]);
                sum = sum + bf16_to_f64(h[e]);
            }
            out[e] = f64_to_bf16_rne(sum * 0.25);
        }
        uint16_t *dst = kblk + (s * (max_ctx / kBlock) + b) * kDI + d8 * 8;
        *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(out);
    }
}

// One thread per (sequence, token, kv head, 4 rotation pairs).  When the
// output is a different buffer the pass-through dims are copied as well.
__global__ void __launch_bounds__(256) kprep_rope_kernel(const uint16_t *__restrict__ k,
                                                         uint16_t *__restrict__ k_rot, int batch,
                                                         int64_t j_lo, int64_t L, int64_t max_ctx,
                                                         RopeFreqs freqs, int copy_rest) {
    constexpr int kQuads = kRD / 2 / 4;  // 8 groups of 4 pairs
    const int64_t per_seq = (L - j_lo) * kHKV * kQuads;
    const int64_t total = per_seq * batch;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t s = i / per_seq;
        int64_t r = i - s * per_seq;
        const int64_t jr = r / (kHKV * kQuads);
        r -= jr * (kHKV * kQuads);
        const int64_t j = j_lo + jr;
        const int g = static_cast<int>(r / kQuads);
        const int qd = static_cast<int>(r - g * kQuads);
        const int64_t row = ((s * max_ctx + j) * kHKV + g) * kD;
        const uint16_t *x = k + row;
        uint16_t *y = k_rot + row;
        const int i0 = qd * 4;
        const uint2 lo = *reinterpret_cast<const uint2 *>(x + i0);
        const uint2 hi = *reinterpret_cast<const uint2 *>(x + i0 + kRD / 2);
        const uint16_t *l16 = reinterpret_cast<const uint16_t *>(&lo);
        const uint16_t *h16 = reinterpret_cast<const uint16_t *>(&hi);
        uint16_t ol[4], oh[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float c, sn;
            rope_cos_sin(j, freqs.inv_freq[i0 + e], c, sn);
            const float x1 = __uint_as_float(static_cast<uint32_t>(l16[e]) << 16);
            const float x2 = __uint_as_float(static_cast<uint32_t>(h16[e]) << 16);
            const float y1 = fmaf(x1, c, -x2 * sn);
            const float y2 = fmaf(x2, c, x1 * sn);
            __nv_bfloat16 b1 = __float2bfloat16_rn(y1), b2 = __float2bfloat16_rn(y2);
            ol[e] = *reinterpret_cast<uint16_t *>(&b1);
            oh[e] = *reinterpret_cast<uint16_t *>(&b2);
        }
        *reinterpret_cast<uint2 *>(y + i0) = *reinterpret_cast<const uint2 *>(ol);
        *reinterpret_cast<uint2 *>(y + i0 + kRD / 2) = *reinterpret_cast<const uint2 *>(oh);
        if (copy_rest) {
            // dims [64, 256): 192 values = 24 x 16 B, split over the 8 quad threads
            const uint4 *src = reinterpret_cast<const uint4 *>(x + kRD);
            uint4 *dst = reinterpret_cast<uint4 *>(y + kRD);
#pragma unroll
            for (int e = qd; e < (kD - kRD) / 8; e += kQuads) dst[e] = src[e];
        }
    }
}

static int grid_for(int64_t work, int threads, int sms) {
    int64_t g = (work + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sms) * 16;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return static_cast<int>(g);
}

cudaError_t launch_kprep(int batch, int64_t t_begin, int64_t L, int64_t max_ctx, const uint16_t *ki,
                         const uint16_t *k, uint16_t *k_rot, uint16_t *kblk,
                         const RopeFreqs &freqs, int sms, cudaStream_t stream) {
    const int64_t nb = L / kBlock;
    const int64_t b_lo = t_begin / kBlock;
    if (nb > b_lo && ki && kblk) {
        const int64_t work = (nb - b_lo) * (kDI / 8) * batch;
        kprep_blocks_kernel<<<grid_for(work, 256, sms), 256, 0, stream>>>(ki, kblk, batch, b_lo, nb,
                                                                          max_ctx);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (k && k_rot && L > t_begin) {
        const int64_t work = (L - t_begin) * kHKV * 8 * batch;
        kprep_rope_kernel<<<grid_for(work, 256, sms), 256, 0, stream>>>(
            k, k_rot, batch, t_begin, L, max_ctx, freqs, k != k_rot ? 1 : 0);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace qsa
