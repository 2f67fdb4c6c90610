// Block-level building blocks shared by the per-row and per-request kernels: radix
// selection of the k-th largest 32-bit key, bitonic sort of 64-bit keys, deterministic
// scans and sums in double precision.  All are fixed-order, so results do not depend on
// scheduling.
#pragma once

#include "dspark_internal.cuh"

namespace dspark {

// k-th largest (1-based, with multiplicity) of keys[0..n) in shared memory; 0 < k <= n.
// Four passes of 8 bits from the top; hist is 256 ints of shared memory.
__device__ inline uint32_t block_kth_largest_key(const uint32_t* keys, int n, int k, int* hist, int* s_bcast) {
    const int tid = threadIdx.x, nt = blockDim.x;
    uint32_t prefix = 0, pmask = 0;
    int kk = k;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < 256; i += nt) hist[i] = 0;
        __syncthreads();
        for (int i = tid; i < n; i += nt) {
            const uint32_t key = keys[i];
            if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
        }
        __syncthreads();
        if (tid < 32) {
            // lane l owns digits 255-8l .. 248-8l (descending)
            int c[8], s = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) { c[q] = hist[255 - 8 * tid - q]; s += c[q]; }
            int incl = s;
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o) incl += y;
            }
            const int excl = incl - s;
            const bool here = excl < kk && incl >= kk;
            if (here) {
                int run = excl;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (run + c[q] >= kk) {
                        s_bcast[0] = 255 - 8 * tid - q;
                        s_bcast[1] = kk - run;
                        break;
                    }
                    run += c[q];
                }
            }
        }
        __syncthreads();
        const uint32_t digit = static_cast<uint32_t>(s_bcast[0]);
        kk = s_bcast[1];
        prefix |= digit << shift;
        pmask |= 255u << shift;
        __syncthreads();
    }
    return prefix;
}

// Bitonic sort, descending, of keys[0..P) in shared memory (P a power of two).
__device__ inline void block_bitonic_desc(unsigned long long* keys, int P) {
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            __syncthreads();
            for (int i = tid; i < P / 2; i += nt) {
                const int lo = 2 * i - (i & (stride - 1));
                const int hi = lo + stride;
                const bool desc = ((lo & size) == 0);
                const unsigned long long a = keys[lo], b = keys[hi];
                if ((a < b) == desc) { keys[lo] = b; keys[hi] = a; }
            }
        }
    }
    __syncthreads();
}

__device__ inline int next_pow2(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

// Exclusive scan in double of vals[0..n) (n <= 4*blockDim.x) into excl[0..n]; excl[n] = total.
// Fixed order: four consecutive elements per thread, warp shuffles, then warp totals in order.
// excl may alias vals.
__device__ inline void block_scan_excl_d(const double* vals, double* excl, int n, double* s_warp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int i0 = 4 * tid;
    double v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = i0 + q < n ? vals[i0 + q] : 0.0;
    const double s = (v[0] + v[1]) + (v[2] + v[3]);
    double incl = s;
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    __syncthreads();
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (tid == 0) {
        double run = 0.0;
        for (int w = 0; w < nw; ++w) { const double t = s_warp[w]; s_warp[w] = run; run += t; }
        s_warp[nw] = run;
    }
    __syncthreads();
    double base = s_warp[warp] + (incl - s);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (i0 + q < n) excl[i0 + q] = base;
        base += v[q];
    }
    if (tid == 0) excl[n] = s_warp[nw];
    __syncthreads();
}

// Sum in double with a fixed order (per-thread strided partials, warp shuffles, warps in order).
__device__ inline double block_sum_d(double v, double* s_warp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    v = warp_sum_d(v);
    __syncthreads();
    if (lane == 0) s_warp[warp] = v;
    __syncthreads();
    if (tid == 0) {
        double t = 0.0;
        for (int w = 0; w < nw; ++w) t += s_warp[w];
        s_warp[nw] = t;
    }
    __syncthreads();
    const double r = s_warp[nw];
    __syncthreads();
    return r;
}

__device__ inline float block_max_nan(float v, float* s_warp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    for (int o = 16; o; o >>= 1) {
        const float y = __shfl_xor_sync(0xffffffffu, v, o);
        v = (v != v || y != y) ? __int_as_float(0x7fc00000) : fmaxf(v, y);
    }
    __syncthreads();
    if (lane == 0) s_warp[warp] = v;
    __syncthreads();
    float r = s_warp[0];
    for (int w = 1; w < nw; ++w) {
        const float y = s_warp[w];
        r = (r != r || y != y) ? __int_as_float(0x7fc00000) : fmaxf(r, y);
    }
    __syncthreads();
    return r;
}

__device__ inline int block_min_i(int v, int* s_warp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    v = warp_min_i(v);
    __syncthreads();
    if (lane == 0) s_warp[warp] = v;
    __syncthreads();
    int r = s_warp[0];
    for (int w = 1; w < nw; ++w) r = min(r, s_warp[w]);
    __syncthreads();
    return r;
}

__device__ inline int block_or_i(int v, int* s_warp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    for (int o = 16; o; o >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if (lane == 0) s_warp[warp] = v;
    __syncthreads();
    int r = 0;
    for (int w = 0; w < nw; ++w) r |= s_warp[w];
    __syncthreads();
    return r;
}

}  // namespace dspark
