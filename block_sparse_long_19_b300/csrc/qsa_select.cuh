// Exact top-k selection helpers (warp level, items held in registers).
//
// Order used everywhere: score descending, then block index ascending.  A
// score is mapped to an order-preserving 32-bit key (larger float -> larger
// key); ties on the key are broken by the block index.
//
// The radix passes only look at the bits below the prefix that all candidate
// keys share (found with a warp max/min): candidate lists hold the best
// scores seen so far, whose keys agree on their top bits, so a histogram of
// the top byte would put every item into one bin.
#pragma once

#include "qsa_common.cuh"

namespace qsa {

struct RadixOut {
    uint32_t thr;  // threshold value (bits below `lo` are zero)
    int krem;      // items still needed from the bucket [thr, thr + 2^lo)
    int eq;        // items in that bucket
    int lo;        // 0: thr is an exact value
};

// Finds, among the items i with bit i of `vm` set (item i of this lane),
// a bucket [thr, thr + 2^lo) that holds the k-th largest value, spending at
// most `max_passes` 8-bit digit passes (or until the bucket holds exactly
// the items still needed).  Requires 1 <= k <= number of valid items.
// hist: 256 words of shared memory owned by this warp.
// NEG: rank ~v instead of v (used to prefer lower block indices).
template <int NI, bool NEG = false>
__device__ __forceinline__ RadixOut warp_radix(const uint32_t (&vin)[NI], uint32_t vm, int k,
                                               int max_passes, uint32_t *hist, int lane) {
    auto v = [&](int i) { return NEG ? ~vin[i] : vin[i]; };
    uint32_t mx = 0u, mn = 0xFFFFFFFFu;
    int nv = 0;
#pragma unroll
    for (int i = 0; i < NI; ++i)
        if ((vm >> i) & 1u) {
            mx = max(mx, v(i));
            mn = min(mn, v(i));
            ++nv;
        }
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    mn = __reduce_min_sync(0xFFFFFFFFu, mn);
    nv = __reduce_add_sync(0xFFFFFFFFu, nv);
    RadixOut r;
    r.krem = k;
    if (mx == mn) {
        r.thr = mx;
        r.eq = nv;
        r.lo = 0;
        return r;
    }
    const int hi = 32 - __clz(mx ^ mn);  // bits [hi, 32) are shared by every item
    unsigned long long prefix = hi >= 32 ? 0ull : (static_cast<unsigned long long>(mx >> hi) << hi);
    int lo = hi;
    int eq = nv;
    for (int pass = 0; pass < max_passes && lo > 0; ++pass) {
        const int w = lo >= 8 ? 8 : lo;
        lo -= w;
        const uint32_t dmask = (1u << w) - 1u;
#pragma unroll
        for (int b = 0; b < 8; ++b) hist[lane * 8 + b] = 0u;
        __syncwarp();
        const unsigned long long want = prefix >> (lo + w);
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            if (((vm >> i) & 1u) && ((static_cast<unsigned long long>(v(i)) >> (lo + w)) == want))
                atomicAdd(&hist[(v(i) >> lo) & dmask], 1u);
        }
        __syncwarp();
        // lane l owns digits 255-8l .. 248-8l (descending)
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
        const bool mine = excl < static_cast<uint32_t>(r.krem) && static_cast<uint32_t>(r.krem) <= incl;
        int digit = 0;
        uint32_t above = 0, e = 0;
        if (mine) {
            uint32_t acc = excl;
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                if (acc + cnt[b] >= static_cast<uint32_t>(r.krem)) {
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
        r.krem -= static_cast<int>(above);
        eq = static_cast<int>(e);
        prefix |= static_cast<unsigned long long>(digit) << lo;
        __syncwarp();
        if (eq == r.krem) break;  // the whole bucket is in: [prefix, prefix + 2^lo) is exact
    }
    r.thr = static_cast<uint32_t>(prefix);
    r.eq = eq;
    r.lo = lo;
    return r;
}

// Exact selection of the k best (key desc, block asc) among the valid
// items; sets bit i of the returned mask for every selected item of this
// lane.  Also returns the streaming threshold a later (higher-index) block
// must reach to enter the selected set: s >= *theta.
template <int NI>
__device__ __forceinline__ uint32_t warp_select_exact(const uint32_t (&key)[NI],
                                                      const uint32_t (&blk)[NI], uint32_t vm,
                                                      int k, uint32_t *hist, int lane,
                                                      float *theta) {
    const RadixOut r = warp_radix<NI>(key, vm, k, 8, hist, lane);
    uint32_t sel = 0;
    if (r.eq == r.krem) {
        // every item of the final bucket is in
#pragma unroll
        for (int i = 0; i < NI; ++i)
            if (((vm >> i) & 1u) && key[i] >= r.thr) sel |= 1u << i;
        *theta = r.lo == 0 ? nextafterf(key2f(r.thr), INFINITY) : key2f(r.thr);
        return sel;
    }
    // r.lo == 0: the k-th key is exactly r.thr and only r.krem of its r.eq
    // copies are taken -- the ones with the lowest block index
    uint32_t vm2 = 0;
#pragma unroll
    for (int i = 0; i < NI; ++i)
        if (((vm >> i) & 1u) && key[i] == r.thr) vm2 |= 1u << i;
    const RadixOut r2 = warp_radix<NI, true>(blk, vm2, r.krem, 8, hist, lane);
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        if (!((vm >> i) & 1u)) continue;
        if (key[i] > r.thr || (key[i] == r.thr && ~blk[i] >= r2.thr)) sel |= 1u << i;
    }
    *theta = nextafterf(key2f(r.thr), INFINITY);
    return sel;
}

// Ascending bitonic sort of 512 distinct keys held by 128 threads (four
// whole warps that share hardware barrier `bar`), thread tg holding
// positions 4tg .. 4tg+3.  Partners one or two positions away are in the
// same thread, up to 64 away in the same warp
// (shuffles); the three steps that cross warps go through shared memory,
// alternating between buf[0..511] and buf[512..1023].  The caller's input may
// sit in buf[512..1023]: the first write there comes after the barrier of
// the first crossing step, which every thread reaches with its keys loaded.
template <typename T>
__device__ __forceinline__ void group_sort512(T (&v)[4], T *buf, int tg, int bar) {
    int flip = 0;
#pragma unroll
    for (int k = 2; k <= 512; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j >= 1; j >>= 1) {
            if (j < 4) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    if (r & j) continue;
                    const int e = 4 * tg + r;
                    const bool asc = (e & k) == 0;
                    const T lo = v[r], hi = v[r ^ j];
                    const bool sw = asc ? (lo > hi) : (lo < hi);
                    v[r] = sw ? hi : lo;
                    v[r ^ j] = sw ? lo : hi;
                }
            } else {
                T o[4];
                if (j >= 128) {
                    T *b = buf + (flip & 1) * 512;
                    ++flip;
#pragma unroll
                    for (int r = 0; r < 4; ++r) b[4 * tg + r] = v[r];
                    asm volatile("bar.sync %0, 128;" ::"r"(bar) : "memory");
                    const int pt = tg ^ (j >> 2);
#pragma unroll
                    for (int r = 0; r < 4; ++r) o[r] = b[4 * pt + r];
                } else {
#pragma unroll
                    for (int r = 0; r < 4; ++r) o[r] = __shfl_xor_sync(0xFFFFFFFFu, v[r], j >> 2);
                }
                const int e = 4 * tg;
                const bool keep_min = ((e & j) == 0) == ((e & k) == 0);
#pragma unroll
                for (int r = 0; r < 4; ++r) v[r] = keep_min ? min(v[r], o[r]) : max(v[r], o[r]);
            }
        }
    }
}

}  // namespace qsa
