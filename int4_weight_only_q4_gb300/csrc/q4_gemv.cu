// int4 group-128 weight-only GEMV / skinny GEMM (batch 1..8) for GB300, sm_103a.
//
// What is computed (rumik-oss-1 int4 engine page, rtts.neoandmatrix.me,
// "Step 3" and "Step 7"): Y[b, n] = sum_k (code[n,k] * scale[n,g] + min[n,g]) * X[b,k],
// g = k / 128, fp32 accumulation.  Every group is evaluated as
//     scale * (sum_k code_k x_k)  +  min * (sum_k x_k).
// The page's CUDA kernel turns a code into a float without a conversion by
// placing it in the mantissa of an fp16 with a fixed exponent (1024 + code).
// Here the codes become bf16 operands with a single AND per two codes and no
// offset at all: a bf16 whose exponent field is 0 or 1 and whose low 8 bits
// hold m has the value m * 2^-133 exactly, so (w & 0x000F000F) is two codes
// and (w & 0x00F000F0) two codes times 16.  The activations are staged times
// a per-column power of two (and 1/16 for the high nibbles) that keeps every
// product a normal fp32 number, and the group sum is multiplied back.  No
// offset means the accumulator carries only the result (an offset of 128
// would make it carry 128 * sum(x) and lose ~4 bits).
//
// The dot products of a 16-row tile and one group run on the tensor cores:
// eight mma.m16n8k16 (16 rows x 8 batch columns x 16 k), bf16 in, fp32
// accumulators; batch columns b >= B are zero.  Because the tensor core
// computes each output column from its own column of the B operand, column b
// is the same whatever the other columns hold.
//
// Weight layouts.  The canonical layout L0 (include/q4.h) is what the export
// job writes.  For streaming, each matrix also gets a tiled copy L1 built once
// on the device (q4_tile): for every 16-row tile j and 128-column group g one
// contiguous 1,088-byte record
//     [  0, 512)  lane l's 16 code bytes of row 16j + l/4, columns 32(l%4)..+31
//     [512,1024)  the same for row 16j + l/4 + 8
//     [1024,1088) for q = 0..7: scale|min<<16 of row 16j+q, then of row 16j+q+8
// records ordered tile-major (j, then g).  A warp reads a record with two
// 512-byte loads and one 64-byte load, all contiguous; a CTA's rows are one
// contiguous byte range; a run of groups of one tile is one bulk copy.
//
// Work split (depends on N, K and the SM count only -- never on B): CTA
// (rb, ks) owns a block of rows (whole 16-row tiles for L1) and groups
// [G*ks/KS, G*(ks+1)/KS).  Inside a CTA the (tile, group) units are dealt to
// the warps in contiguous ranges (direct kernel) or streamed in chunks of 8
// groups (stream kernel); partial sums are added in a fixed order (warp order
// or chunk order), and with KS > 1 the CTA results go to the workspace and
// the last CTA of the row block (arrival ticket) adds them in k-split order.
// Every addition order is therefore fixed by (N, K, SMs), which makes each
// batch column bit-identical to the batch-1 result (the pure-C TTS engine
// page, wpnews.pro: match the accumulation order).
//
// Kernels.  "direct": one CTA per SM, persistent over a list of matrices;
// every lane loads its codes straight into registers DEPTH units ahead, and
// the first units of the next matrix are in flight while the current one is
// being finished.  "stream": a producer warp streams chunks of L1 records with
// 1-D bulk copies (cp.async.bulk) into a shared-memory ring guarded by
// mbarriers; consumer warp w owns stages w, w+W, ..., w+(D-1)W and takes every
// W-th chunk, so it waits for a round of a stage only after it has released
// the previous round itself and the mbarrier phase parity cannot alias.
// Both stage the activations per matrix in shared memory in B-fragment order
// with the per-group sums of x.
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "q4.h"
#include "q4_common.cuh"

namespace {

constexpr int kMaxB = 8;
constexpr int64_t kMaxK = 65536;
constexpr int kMaxDevices = 64;
constexpr size_t kSmemLimit = 220 * 1024;  // dynamic; leaves room for static smem under the 227 KB cap

constexpr int kRecBytes = 1088;                 // one L1 record: 16 rows x 128 columns + scale/min
constexpr int kRec8Bytes = 2048;  // int8 head record: 16 rows x 128 codes
constexpr int kKC = 8;                          // groups (records) per streamed chunk
constexpr int kStageBytes = kKC * kRecBytes;    // one stream-ring stage
constexpr int kMaxMats = 128;                   // matrices per stream launch (kernel parameter table)
constexpr int kHdrBytes = 512;                  // ring header: up to 2 x 24 mbarriers + the k-split flag
constexpr unsigned kDefaultWaitLimit = 1u << 22;

// Device-side error word: bit 0 = a bounded barrier wait gave up.
__device__ unsigned int g_q4_device_error;

// ------------------------------------------------------------------ device helpers
__device__ __forceinline__ uint4 ld_stream_u4(const uint8_t* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint2 ld_stream_u2(const uint8_t* p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_nc_u16(const uint16_t* p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float half_bits_to_f32(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
}


// Ask L2 to fetch [p, p + bytes) from DRAM (bytes: multiple of 16, p: 16-byte aligned).
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// wait_group with a run-time count n in [0, N]
template <int N>
__device__ __forceinline__ void cp_async_wait_upto(int n) {
    if constexpr (N == 0) {
        cp_async_wait<0>();
    } else {
        if (n >= N) cp_async_wait<N>();
        else cp_async_wait_upto<N - 1>(n);
    }
}

__device__ __forceinline__ void report_timeout() { atomicOr(&g_q4_device_error, 1u); }

__device__ __forceinline__ uint4 lds128(const unsigned char* p) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(smem_addr(p)));
    return r;
}

__device__ __forceinline__ uint4 lds128_s(uint32_t a) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a));
    return r;
}
__device__ __forceinline__ uint2 lds64_s(uint32_t a) {
    uint2 r;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(a));
    return r;
}
__device__ __forceinline__ void cp_async16_s(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ uint2 lds64(const unsigned char* p) {
    uint2 r;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(smem_addr(p)));
    return r;
}

template <int NTHREADS>
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(NTHREADS) : "memory");
}

// ------------------------------------------------------------------ one 16-row x 128-column group
// Codes as bf16 operands without arithmetic: a bf16 whose exponent field is 0 or 1 and whose
// low 8 bits hold m is exactly m * 2^-133 (the subnormals continue into the first normal
// binade with the same spacing).  So w & 0x000F000F is the bf16 pair {c0, c4} * 2^-133 and
// w & 0x00F000F0 is {c1, c5} * 16 * 2^-133 -- one LOP3 per two codes, no offset to remove.
// The activations are staged multiplied by 2^a (paired with low nibbles) or 2^(a-4) (paired
// with high nibbles), a chosen per batch column so the products stay normal fp32 numbers, and
// the epilogue multiplies the group sum by 2^(133-a).  Every step is exact except the fp32
// additions.
__device__ __forceinline__ uint32_t lo_nibbles(uint32_t v) { return v & 0x000F000Fu; }
__device__ __forceinline__ uint32_t hi_nibbles(uint32_t v) { return v & 0x00F000F0u; }

// Fragment-order x: entry (group gl, word i, half p, lane 4n+t), BT entries per lane quad.
template <int BT>
__device__ __forceinline__ size_t xfrag_index(int gl, int i, int p) {
    return (static_cast<size_t>(gl) * 8 + i * 2 + p) * (4 * BT);
}

template <bool GLOBAL>
__device__ __forceinline__ uint2 ld_x(const uint2* p) {
    if constexpr (GLOBAL) return ld_dep_u2(p);
    return *p;
}

// qa/qb: this lane's 32 codes (16 bytes) of tile rows q and q+8, columns 32t..32t+31 of the group.
// xg: the group's staged activations.  c: rows (q, q, q+8, q+8) x batch columns (2t, 2t+1, 2t,
// 2t+1) of sum_k code * x * 2^(a-133).
template <bool MMA, int BT, bool XG = false>
__device__ __forceinline__ void group_dot(const uint4& qa, const uint4& qb, const uint2* xg, int lane, int B,
                                          float (&c)[4]) {
    const int t = lane & 3, q = lane >> 2;
    const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w};
    const uint32_t wb[4] = {qb.x, qb.y, qb.z, qb.w};
    c[0] = c[1] = c[2] = c[3] = 0.f;
    if constexpr (MMA) {
        const bool xon = q < B;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // word i holds columns 8i..8i+7 of the lane's 32: pairs (0,4) (1,5) | (2,6) (3,7)
            const uint32_t wa8 = wa[i] >> 8, wb8 = wb[i] >> 8;
            uint2 x0 = make_uint2(0, 0), x1 = make_uint2(0, 0);
            if (xon) {
                x0 = ld_x<XG>(xg + xfrag_index<BT>(0, i, 0) + lane);
                x1 = ld_x<XG>(xg + xfrag_index<BT>(0, i, 1) + lane);
            }
            mma_bf16_m16n8k16(c, lo_nibbles(wa[i]), lo_nibbles(wb[i]), hi_nibbles(wa[i]), hi_nibbles(wb[i]), x0.x,
                              x0.y);
            mma_bf16_m16n8k16(c, lo_nibbles(wa8), lo_nibbles(wb8), hi_nibbles(wa8), hi_nibbles(wb8), x1.x, x1.y);
        }
    } else {
        float pa[BT], pb[BT];
#pragma unroll
        for (int n = 0; n < BT; ++n) { pa[n] = 0.f; pb[n] = 0.f; }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                const uint32_t va = wa[i] >> (8 * p), vb = wb[i] >> (8 * p);
                const uint32_t A0 = lo_nibbles(va), A1 = hi_nibbles(va);
                const uint32_t B0 = lo_nibbles(vb), B1 = hi_nibbles(vb);
                const float a00 = bf16lo_to_f32(A0), a01 = bf16hi_to_f32(A0);
                const float a10 = bf16lo_to_f32(A1), a11 = bf16hi_to_f32(A1);
                const float b00 = bf16lo_to_f32(B0), b01 = bf16hi_to_f32(B0);
                const float b10 = bf16lo_to_f32(B1), b11 = bf16hi_to_f32(B1);
#pragma unroll
                for (int n = 0; n < BT; ++n) {
                    uint2 xv = make_uint2(0, 0);
                    if (n < B) xv = ld_x<XG>(xg + xfrag_index<BT>(0, i, p) + n * 4 + t);
                    const float x00 = bf16lo_to_f32(xv.x), x01 = bf16hi_to_f32(xv.x);
                    const float x10 = bf16lo_to_f32(xv.y), x11 = bf16hi_to_f32(xv.y);
                    pa[n] = fmaf(a00, x00, pa[n]);
                    pa[n] = fmaf(a01, x01, pa[n]);
                    pa[n] = fmaf(a10, x10, pa[n]);
                    pa[n] = fmaf(a11, x11, pa[n]);
                    pb[n] = fmaf(b00, x00, pb[n]);
                    pb[n] = fmaf(b01, x01, pb[n]);
                    pb[n] = fmaf(b10, x10, pb[n]);
                    pb[n] = fmaf(b11, x11, pb[n]);
                }
            }
        }
        // add the quad's four 32-column pieces; every lane of the quad gets the same value
#pragma unroll
        for (int n = 0; n < BT; ++n) {
            pa[n] += __shfl_xor_sync(0xffffffffu, pa[n], 1);
            pa[n] += __shfl_xor_sync(0xffffffffu, pa[n], 2);
            pb[n] += __shfl_xor_sync(0xffffffffu, pb[n], 1);
            pb[n] += __shfl_xor_sync(0xffffffffu, pb[n], 2);
        }
#pragma unroll
        for (int n = 0; n < BT; ++n) {
            if (n == 2 * t) { c[0] = pa[n]; c[2] = pb[n]; }
            if (n == 2 * t + 1) { c[1] = pa[n]; c[3] = pb[n]; }
        }
    }
}

// The tensor-core dot of one group with this lane's activation fragments in registers (xv[i] =
// fragments (i, 0) and (i, 1)) as two independent mma chains (words 0-1 and 2-3) added at the
// end: a fixed order, half the dependent-mma latency.
__device__ __forceinline__ void group_dot_x4(const uint4& qa, const uint4& qb, const uint4 (&xv)[4],
                                             float (&c)[4]) {
    const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w};
    const uint32_t wb[4] = {qb.x, qb.y, qb.z, qb.w};
    float c2[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float (&d)[4] = (i < 2) ? c : c2;
        const uint32_t wa8 = wa[i] >> 8, wb8 = wb[i] >> 8;
        if (i == 0 || i == 2)
            mma_bf16_m16n8k16_zc(d, lo_nibbles(wa[i]), lo_nibbles(wb[i]), hi_nibbles(wa[i]), hi_nibbles(wb[i]),
                                 xv[i].x, xv[i].y);
        else
            mma_bf16_m16n8k16(d, lo_nibbles(wa[i]), lo_nibbles(wb[i]), hi_nibbles(wa[i]), hi_nibbles(wb[i]),
                              xv[i].x, xv[i].y);
        mma_bf16_m16n8k16(d, lo_nibbles(wa8), lo_nibbles(wb8), hi_nibbles(wa8), hi_nibbles(wb8), xv[i].z, xv[i].w);
    }
    c[0] += c2[0];
    c[1] += c2[1];
    c[2] += c2[2];
    c[3] += c2[3];
}

// acc += scale * (c * f) + min * S for rows q (scale/min packed in sa_ma) and q+8 (sb_mb);
// f = 2^(133-a) of batch columns 2t, 2t+1 undoes the staging scale.
template <bool XG = false>
__device__ __forceinline__ void group_epilogue(float (&acc)[4], const float (&c)[4], uint32_t sa_ma,
                                               uint32_t sb_mb, const float* S2, float f0, float f1) {
    float2 S;
    if constexpr (XG) {
        const uint2 v = ld_dep_u2(S2);
        S = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
    } else {
        S = *reinterpret_cast<const float2*>(S2);
    }
    const float sa = half_bits_to_f32(sa_ma), ma = half_bits_to_f32(sa_ma >> 16);
    const float sb = half_bits_to_f32(sb_mb), mb = half_bits_to_f32(sb_mb >> 16);
    acc[0] = fmaf(sa, c[0] * f0, acc[0]);
    acc[0] = fmaf(ma, S.x, acc[0]);
    acc[1] = fmaf(sa, c[1] * f1, acc[1]);
    acc[1] = fmaf(ma, S.y, acc[1]);
    acc[2] = fmaf(sb, c[2] * f0, acc[2]);
    acc[2] = fmaf(mb, S.x, acc[2]);
    acc[3] = fmaf(sb, c[3] * f1, acc[3]);
    acc[3] = fmaf(mb, S.y, acc[3]);
}

// Stage x[:, 128*g0 .. 128*(g0+Gs)) for the mma B fragments, with the group sums of x and the
// per-column factors: column n gets a_n = 120 - e_n (e_n = exponent of the largest |x| of the
// column's slice, a_n in [6, 253]); entries pairing with low nibbles hold x * 2^a_n, with high
// nibbles x * 2^(a_n-4), and fac[n] = 2^(133 - a_n).  Exact for |x| < 2^121.  S[gl][n] = sum over
// the group (fixed order: 8 sequential adds, then a 16-lane xor tree).
// Entry (gl, i, p, lane = 4n + t) (8 bytes) holds x[n][k], k = 128(g0+gl) + 32t + 8i + {2p, 2p+4,
// 2p+1, 2p+5}: in xfrag order (shared memory of the kernels that compute from it), or with LM
// (prepared copies) entries (gl, i, 0) and (gl, i, 1) of lane L as one 16-byte word, uint4
// (gl * 4 + i) * 4BT + L, so that each of a warp's four loads per group is one contiguous run,
// and the group sums stored already divided by fac (S * 2^(a_n-133), an exact power-of-two
// scaling).  X8 (with LM, for the int8 head): the k pairing of the int8 operands instead -- word
// i of lane (n, t) holds mma 2i and 2i+1, each as (x[k], x[k+2]) | (x[k+1], x[k+3]) with
// k = 32t + 4m for mma m -- and no high-nibble factor.
// A thread's pieces of x are loaded U at a time before any is used (they do not depend on one
// another, so a thread waits for memory once per U pieces); the column maxima are reduced over the
// 16 lanes of a (group, column) before one shared atomic; when every piece fits in one round the
// second pass reuses the registers.  Every thread in [0, nthr) calls this (nthr a multiple of 32);
// sync is the callers' barrier over those threads; colmax: 8 words of scratch shared memory.
template <int BT, bool LM, bool X8, int U, typename Sync>
__device__ __forceinline__ void stage_x_batched(const uint16_t* x, int K, int B, int g0, int Gs, uint2* xs,
                                                float* ssum, float* fac, unsigned* colmax, int tid, int nthr,
                                                Sync sync) {
    const int items = Gs * B * 16;  // (group, column, chunk t, word i); (t, i) fastest
    // gn / B as a multiply and shift: exact for gn < 2^16 (gn < G B <= 4096 here), and the product
    // stays below 2^32 for gn < 2^13
    const uint32_t binv = (1u << 19) / B + ((1u << 19) % B != 0 ? 1u : 0u);
    auto div_b = [&](int gn) { return static_cast<int>((static_cast<uint32_t>(gn) * binv) >> 19); };
    auto piece = [&](int idx) -> uint4 {
        const int ti = idx & 15, gn = idx >> 4;
        const int gl = div_b(gn), n = gn - gl * B;
        return *reinterpret_cast<const uint4*>(x + static_cast<size_t>(n) * K + static_cast<size_t>(g0 + gl) * 128 +
                                               (ti >> 2) * 32 + (ti & 3) * 8);
    };
    if (tid < 8) colmax[tid] = 0u;
    sync();
    uint4 v[U];
    for (int r0 = 0; r0 < items; r0 += U * nthr) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int idx = r0 + u * nthr + tid;
            v[u] = idx < items ? piece(idx) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (r0 + u * nthr >= items) break;  // the same for every thread
            const int idx = r0 + u * nthr + tid;
            const uint32_t h[8] = {v[u].x << 16, v[u].x & 0xFFFF0000u, v[u].y << 16, v[u].y & 0xFFFF0000u,
                                   v[u].z << 16, v[u].z & 0xFFFF0000u, v[u].w << 16, v[u].w & 0xFFFF0000u};
            uint32_t mx = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) mx = max(mx, h[e] & 0x7FFFFFFFu);
            float s = bf16lo_to_f32(v[u].x);
            s += bf16hi_to_f32(v[u].x);
            s += bf16lo_to_f32(v[u].y);
            s += bf16hi_to_f32(v[u].y);
            s += bf16lo_to_f32(v[u].z);
            s += bf16hi_to_f32(v[u].z);
            s += bf16lo_to_f32(v[u].w);
            s += bf16hi_to_f32(v[u].w);
            // the 16 lanes of one (group, column): items are whole multiples of 16, so these lanes
            // are all in range or all out of it
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) {
                mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                s += __shfl_xor_sync(0xffffffffu, s, o);
            }
            if (idx < items && (idx & 15) == 0) {
                const int gn = idx >> 4;
                const int gl = div_b(gn), n = gn - gl * B;
                atomicMax(&colmax[n], mx);
                ssum[gl * 8 + n] = s;
            }
        }
    }
    for (int idx = tid; idx < Gs * 8; idx += nthr)
        if ((idx & 7) >= B) ssum[idx] = 0.f;
    sync();
    const bool one_round = items <= U * nthr;
    for (int r0 = 0; r0 < items; r0 += U * nthr) {
        if (!one_round) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int idx = r0 + u * nthr + tid;
                v[u] = idx < items ? piece(idx) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int idx = r0 + u * nthr + tid;
            if (idx >= items) break;
            const int ti = idx & 15, gn = idx >> 4;
            const int gl = div_b(gn), n = gn - gl * B;
            const int tt = ti >> 2, i = ti & 3;
            const int e = static_cast<int>(colmax[n] >> 23) - 127;  // colmax == 0: e = -127
            int a = 120 - e;
            a = a < 6 ? 6 : (a > 253 ? 253 : a);
            // x * 2^a as two exact power-of-two products, so that 2^a itself need not be a float
            const int a1 = a > 127 ? 127 : a;
            const float m1 = __int_as_float((a1 + 127) << 23);
            const float m2 = __int_as_float((a - a1 + 127) << 23);
            uint2 p0, p1;
            if constexpr (X8) {
                p0.x = bf16x2_scale(__byte_perm(v[u].x, v[u].y, 0x5410), m1, m2);
                p0.y = bf16x2_scale(__byte_perm(v[u].x, v[u].y, 0x7632), m1, m2);
                p1.x = bf16x2_scale(__byte_perm(v[u].z, v[u].w, 0x5410), m1, m2);
                p1.y = bf16x2_scale(__byte_perm(v[u].z, v[u].w, 0x7632), m1, m2);
            } else {
                p0.x = bf16x2_scale(__byte_perm(v[u].x, v[u].z, 0x5410), m1, m2);
                p0.y = bf16x2_scale(__byte_perm(v[u].x, v[u].z, 0x7632), m1, m2 * 0.0625f);
                p1.x = bf16x2_scale(__byte_perm(v[u].y, v[u].w, 0x5410), m1, m2);
                p1.y = bf16x2_scale(__byte_perm(v[u].y, v[u].w, 0x7632), m1, m2 * 0.0625f);
            }
            if constexpr (LM) {
                const size_t li = (static_cast<size_t>(gl) * 4 + i) * 4 * BT + n * 4 + tt;
                reinterpret_cast<uint4*>(xs)[li] = make_uint4(p0.x, p0.y, p1.x, p1.y);
                if (ti == 0) {  // this thread wrote ssum[gl * 8 + n] in the first pass
                    const int es = a - 133, e1 = es < -63 ? -63 : es, e2 = es - e1;
                    ssum[gl * 8 + n] = (ssum[gl * 8 + n] * __int_as_float((e1 + 127) << 23)) *
                                       __int_as_float((e2 + 127) << 23);
                }
            } else {
                const size_t base = xfrag_index<BT>(gl, i, 0) + n * 4 + tt;
                xs[base] = p0;
                xs[base + 4 * BT] = p1;
            }
        }
    }
    if (tid < 8) {
        const int e = static_cast<int>(colmax[tid] >> 23) - 127;
        int a = 120 - e;
        a = a < 6 ? 6 : (a > 253 ? 253 : a);
        fac[tid] = __int_as_float((133 - a + 127) << 23);  // 2^(133-a), 2^-120 .. 2^127
    }
}

// ================================================================== L1 tiled layout
// One thread per 16-byte piece of a record: pieces 0..63 are code bytes, 64..67 scale/min.
__global__ void q4_tile_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                               const uint16_t* __restrict__ mins, int N, int K, uint8_t* __restrict__ tiled,
                               int64_t pieces) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= pieces) return;
    const int G = K >> 7;
    const int64_t rec = idx / 68;
    const int piece = static_cast<int>(idx - rec * 68);
    const int j = static_cast<int>(rec / G);
    const int g = static_cast<int>(rec - static_cast<int64_t>(j) * G);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (piece < 64) {
        const int h = piece >> 5, l = piece & 31;
        const int row = 16 * j + (l >> 2) + 8 * h;
        if (row < N)
            v = *reinterpret_cast<const uint4*>(codes + static_cast<size_t>(row) * (K >> 1) + g * 64 + (l & 3) * 16);
    } else {
        const int pp = piece - 64;  // q = 2pp and 2pp + 1
        uint32_t w[4] = {0, 0, 0, 0};
        for (int e = 0; e < 2; ++e) {
            const int q = 2 * pp + e;
            for (int h = 0; h < 2; ++h) {
                const int row = 16 * j + q + 8 * h;
                if (row < N) {
                    const size_t o = static_cast<size_t>(row) * G + g;
                    w[2 * e + h] = static_cast<uint32_t>(scales[o]) | (static_cast<uint32_t>(mins[o]) << 16);
                }
            }
        }
        v = make_uint4(w[0], w[1], w[2], w[3]);
    }
    *reinterpret_cast<uint4*>(tiled + rec * kRecBytes + piece * 16) = v;
}

// The int8 head's tiled copy: one thread per 16-byte piece of a 2,048-byte record (128 pieces):
// piece 64h + 2l + e holds row 16j + l/4 + 8h, columns 128g + 32(l%4) + 16e .. +15.
__global__ void q8_tile_kernel(const int8_t* __restrict__ codes, int N, int K, uint8_t* __restrict__ tiled,
                               int64_t pieces) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= pieces) return;
    const int G = K >> 7;
    const int64_t rec = idx >> 7;
    const int piece = static_cast<int>(idx & 127);
    const int j = static_cast<int>(rec / G);
    const int g = static_cast<int>(rec - static_cast<int64_t>(j) * G);
    const int h = piece >> 6, l = (piece >> 1) & 31, e = piece & 1;
    const int row = 16 * j + (l >> 2) + 8 * h;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < N)
        v = *reinterpret_cast<const uint4*>(codes + static_cast<size_t>(row) * K + g * 128 + (l & 3) * 32 + e * 16);
    *reinterpret_cast<uint4*>(tiled + rec * kRec8Bytes + h * 1024 + l * 32 + e * 16) = v;
}

// ================================================================== work lists
struct MatDesc {
    const uint8_t* codes;     // L0 (may be null when `tiled` is used)
    const uint16_t* scales;
    const uint16_t* mins;
    const uint8_t* tiled;     // L1 records (may be null for the L0 kernels)
    const uint16_t* x;
    float* y;
    float* ws_part;           // [k_splits][B][N] when k_splits > 1
    unsigned* ws_cnt;         // [row_blocks][passes]
    int N, K;
    int row_blocks, k_splits, tiles_per_pass, passes, smax;
    int rot;                  // CTA c takes row block (c / k_splits + rot) % row_blocks
};

struct Params {
    int n_mats;
    int B;
    unsigned wait_limit;
    int l2_ahead;  // direct kernel on L1: records each warp asks L2 to fetch ahead of its loads (0: off)
    MatDesc m[kMaxMats];
};

struct Share {
    int rb, ks, r0, r1, t0, g0, Gs, T;
};

// The part of matrix m that CTA `cta` computes; false if it has none.  TILE_GRAIN: row blocks
// are whole 16-row tiles (L1); otherwise any rows (L0).
template <bool TILE_GRAIN>
__device__ __forceinline__ bool cta_share(const MatDesc& m, int cta, Share& s) {
    if (cta >= m.row_blocks * m.k_splits) return false;
    const int G = m.K >> 7;
    const int rbx = cta / m.k_splits;
    s.ks = cta - rbx * m.k_splits;
    s.rb = (rbx + m.rot) % m.row_blocks;
    if (TILE_GRAIN) {
        const int T_all = (m.N + 15) >> 4;
        s.t0 = static_cast<int>(static_cast<int64_t>(s.rb) * T_all / m.row_blocks);
        const int t1 = static_cast<int>(static_cast<int64_t>(s.rb + 1) * T_all / m.row_blocks);
        s.r0 = 16 * s.t0;
        s.r1 = min(m.N, 16 * t1);
    } else {
        s.r0 = static_cast<int>(static_cast<int64_t>(s.rb) * m.N / m.row_blocks);
        s.r1 = static_cast<int>(static_cast<int64_t>(s.rb + 1) * m.N / m.row_blocks);
        s.t0 = 0;
    }
    s.g0 = static_cast<int>(static_cast<int64_t>(s.ks) * G / m.k_splits);
    const int g1 = static_cast<int>(static_cast<int64_t>(s.ks + 1) * G / m.k_splits);
    s.Gs = g1 - s.g0;
    s.T = (s.r1 - s.r0 + 15) >> 4;
    return true;
}

struct Stage {
    uint4 qa, qb;            // 32 codes of row q and of row q+8
    uint32_t sa_ma, sb_mb;   // fp16 bits: scale | min << 16
};

// Warp w of WARPS gets units [w*U/WARPS, (w+1)*U/WARPS).
__device__ __forceinline__ int range_begin(int w, int U, int warps) {
    return static_cast<int>((static_cast<int64_t>(w) * U) / warps);
}
// The warp whose range holds unit u.
__device__ __forceinline__ int range_owner(int u, int U, int warps) {
    return static_cast<int>(((static_cast<int64_t>(u) + 1) * warps - 1) / U);
}

template <bool TILED>
__device__ __forceinline__ void load_unit(Stage& s, const MatDesc& m, const Share& sh, int j, int gl, int lane) {
    const int G = m.K >> 7;
    if constexpr (TILED) {
        const uint8_t* rec = m.tiled + (static_cast<size_t>(sh.t0 + j) * G + sh.g0 + gl) * kRecBytes;
        s.qa = ld_stream_u4(rec + 16 * lane);
        s.qb = ld_stream_u4(rec + 512 + 16 * lane);
        const uint2 v = ld_stream_u2(rec + 1024 + 8 * (lane >> 2));
        s.sa_ma = v.x;
        s.sb_mb = v.y;
    } else {
        const int q = lane >> 2, t = lane & 3;
        const size_t row_bytes = static_cast<size_t>(m.K) >> 1;
        const int g = sh.g0 + gl;
        const int ra = sh.r0 + j * 16 + q;
        const int rbw = ra + 8;
        if (ra < sh.r1) {
            s.qa = ld_stream_u4(m.codes + static_cast<size_t>(ra) * row_bytes + g * 64 + t * 16);
            s.sa_ma = ld_nc_u16(m.scales + static_cast<size_t>(ra) * G + g) |
                      (ld_nc_u16(m.mins + static_cast<size_t>(ra) * G + g) << 16);
        } else {
            s.qa = make_uint4(0, 0, 0, 0);
            s.sa_ma = 0;
        }
        if (rbw < sh.r1) {
            s.qb = ld_stream_u4(m.codes + static_cast<size_t>(rbw) * row_bytes + g * 64 + t * 16);
            s.sb_mb = ld_nc_u16(m.scales + static_cast<size_t>(rbw) * G + g) |
                      (ld_nc_u16(m.mins + static_cast<size_t>(rbw) * G + g) << 16);
        } else {
            s.qb = make_uint4(0, 0, 0, 0);
            s.sb_mb = 0;
        }
    }
}

// Final per-row sums of a CTA's share: to Y, or through the workspace (k-split, last CTA adds).
template <int NT, typename Sync>
__device__ __forceinline__ void finish_rows(const MatDesc& m, const Share& s, int pass, int prow0, int prows, int B,
                                            int tid, int* flag, Sync sync) {
    if (m.k_splits <= 1) return;
    __threadfence();
    sync();
    unsigned* cnt = m.ws_cnt + s.rb * m.passes + pass;
    if (tid == 0) *flag = (atomicAdd(cnt, 1u) == static_cast<unsigned>(m.k_splits - 1));
    sync();
    if (*flag) {
        __threadfence();
        for (int idx = tid; idx < prows * B; idx += NT) {
            const int b = idx / prows;
            const int rr = idx - b * prows;
            float sum = 0.f;
            for (int k2 = 0; k2 < m.k_splits; ++k2)
                sum += __ldcg(m.ws_part + (static_cast<size_t>(k2) * B + b) * m.N + prow0 + rr);
            m.y[static_cast<size_t>(b) * m.N + prow0 + rr] = sum;
        }
        if (tid == 0) *cnt = 0u;  // ready for the next call
    }
}

__device__ __forceinline__ void store_row_sum(const MatDesc& m, const Share& s, int b, int row, int B, float v) {
    if (m.k_splits == 1)
        m.y[static_cast<size_t>(b) * m.N + row] = v;
    else
        m.ws_part[(static_cast<size_t>(s.ks) * B + b) * m.N + row] = v;
}

// ================================================================== direct kernel
// Shared memory: x in B-fragment order [Gs*256*B] | x group sums [Gs*8] | warp partials
// [WARPS][smax][16][B].
template <int WARPS, int DEPTH, bool TILED, bool MMA, int BT>
__global__ void __launch_bounds__(WARPS * 32, 1) q4_direct_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int flag;
    constexpr int NT = WARPS * 32;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int t = lane & 3;
    const int q = lane >> 2;
    const int tid = threadIdx.x;
    const int B = p.B;

    Stage st[DEPTH];
    int lt = 0, lg = 0;             // load cursor (tile, local group) of the matrix being loaded
    const uint8_t* lrec = nullptr;  // L1: the record at the cursor
    auto find_next = [&](int from, Share& s) -> int {
        for (int i = from; i < p.n_mats; ++i)
            if (cta_share<TILED>(p.m[i], blockIdx.x, s)) return i;
        return -1;
    };
    int lu = 0, lue = 0;            // unit index at the cursor and the end of this warp's range
    // load the unit at the cursor and advance it (consecutive units are consecutive records
    // except where a tile ends inside a k-split); with one k-split, also ask L2 for the record
    // l2_ahead units further on, so that DRAM sees far more requests than registers can hold
    auto load_next = [&](Stage& sg, const MatDesc& mm, const Share& s) {
        if constexpr (TILED) {
            if (p.l2_ahead > 0 && mm.k_splits == 1 && lane == 0 && lu + p.l2_ahead < lue)
                prefetch_l2_bulk(lrec + static_cast<size_t>(p.l2_ahead) * kRecBytes, kRecBytes);
            ++lu;
            sg.qa = ld_stream_u4(lrec + 16 * lane);
            sg.qb = ld_stream_u4(lrec + 512 + 16 * lane);
            const uint2 v = ld_stream_u2(lrec + 1024 + 8 * q);
            sg.sa_ma = v.x;
            sg.sb_mb = v.y;
            lrec += kRecBytes;
            if (++lg == s.Gs) {
                lg = 0;
                ++lt;
                lrec += static_cast<size_t>((mm.K >> 7) - s.Gs) * kRecBytes;
            }
        } else {
            load_unit<false>(sg, mm, s, lt, lg, lane);
            if (++lg == s.Gs) { lg = 0; ++lt; }
        }
    };
    // issue the first DEPTH loads of this warp's range of matrix i
    auto prologue = [&](int i, const Share& s, int ub, int ue) {
        if (ub < ue) {
            lt = ub / s.Gs;
            lg = ub - lt * s.Gs;
            lu = ub;
            lue = ue;
            if constexpr (TILED) {
                lrec = p.m[i].tiled +
                       (static_cast<size_t>(s.t0 + lt) * (p.m[i].K >> 7) + s.g0 + lg) * kRecBytes;
                // the records between the first loads and the steady-state prefetch front
                if (p.l2_ahead > DEPTH && p.m[i].k_splits == 1 && lane == 0) {
                    const int a = ub + DEPTH, b = min(ue, ub + p.l2_ahead);
                    if (a < b)
                        prefetch_l2_bulk(lrec + static_cast<size_t>(DEPTH) * kRecBytes,
                                         static_cast<uint32_t>((b - a) * kRecBytes));
                }
            }
        }
#pragma unroll
        for (int d = 0; d < DEPTH; ++d)
            if (ub + d < ue) load_next(st[d], p.m[i], s);
    };

    Share cs;
    int ci = find_next(0, cs);
    int cU = 0, cub = 0, cue = 0;
    if (ci >= 0) {
        cU = cs.T * cs.Gs;
        cub = range_begin(warp, cU, WARPS);
        cue = range_begin(warp + 1, cU, WARPS);
        prologue(ci, cs, cub, cue);  // weights are read-only: may run before the previous kernel ends
    }
    grid_dependency_wait();  // x may be the previous kernel's output; y and ws are shared with it
    allow_dependents();

    while (ci >= 0) {
        const MatDesc& m = p.m[ci];
        uint2* xs = reinterpret_cast<uint2*>(smem);
        float* ssum = reinterpret_cast<float*>(smem + static_cast<size_t>(cs.Gs) * 256 * BT);
        float* fac = ssum + cs.Gs * 8;
        unsigned* colmax = reinterpret_cast<unsigned*>(fac + 8);
        float* part = reinterpret_cast<float*>(colmax + 8);
        stage_x_batched<BT, false, false, 1>(m.x, m.K, B, cs.g0, cs.Gs, xs, ssum, fac, colmax, tid, NT,
                                             [] { __syncthreads(); });
        __syncthreads();
        const float f0 = fac[2 * t], f1 = fac[2 * t + 1];

        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        int ct = (cub < cue) ? cub / cs.Gs : 0;
        int cgl = (cub < cue) ? cub - ct * cs.Gs : 0;
        const int first_tile = ct;
        auto flush = [&](int tile) {
            if (tile - first_tile >= m.smax) return;  // cannot happen with a plan from make_plan
            float* pp = part + static_cast<size_t>(warp * m.smax + (tile - first_tile)) * 16 * B;
            const int c0 = 2 * t, c1 = 2 * t + 1;
            if (c0 < B) { pp[q * B + c0] = acc[0]; pp[(q + 8) * B + c0] = acc[2]; }
            if (c1 < B) { pp[q * B + c1] = acc[1]; pp[(q + 8) * B + c1] = acc[3]; }
        };
        for (int u = cub; u < cue; u += DEPTH) {
#pragma unroll
            for (int d = 0; d < DEPTH; ++d) {
                if (u + d < cue) {
                    const Stage cur = st[d];
                    if (u + d + DEPTH < cue) load_next(st[d], m, cs);
                    float cc[4];
                    group_dot<MMA, BT>(cur.qa, cur.qb, xs + xfrag_index<BT>(cgl, 0, 0), lane, B, cc);
                    group_epilogue(acc, cc, cur.sa_ma, cur.sb_mb, ssum + cgl * 8 + 2 * t, f0, f1);
                    if (++cgl == cs.Gs) {
                        flush(ct);
                        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
                        cgl = 0;
                        ++ct;
                    }
                }
            }
        }
        if (cub < cue && cgl != 0) flush(ct);

        // start streaming the next matrix while this one is being finished
        Share ns;
        const int ni = find_next(ci + 1, ns);
        int nU = 0, nub = 0, nue = 0;
        if (ni >= 0) {
            nU = ns.T * ns.Gs;
            nub = range_begin(warp, nU, WARPS);
            nue = range_begin(warp + 1, nU, WARPS);
            prologue(ni, ns, nub, nue);
        }
        __syncthreads();

        // add the warp partials of each tile in warp order
        const int rows = cs.r1 - cs.r0;
        for (int idx = tid; idx < rows * B; idx += NT) {
            const int b = idx / rows;
            const int rr = idx - b * rows;
            const int j = rr >> 4, rl = rr & 15;
            const int wf = range_owner(j * cs.Gs, cU, WARPS);
            const int wl = range_owner(j * cs.Gs + cs.Gs - 1, cU, WARPS);
            float sum = 0.f;
            for (int w = wf; w <= wl; ++w) {
                const int bw = range_begin(w, cU, WARPS);
                if (bw >= range_begin(w + 1, cU, WARPS)) continue;  // empty range
                sum += part[(static_cast<size_t>(w * m.smax + (j - bw / cs.Gs)) * 16 + rl) * B + b];
            }
            store_row_sum(m, cs, b, cs.r0 + rr, B, sum);
        }
        finish_rows<NT>(m, cs, 0, cs.r0, rows, B, tid, &flag, [] { __syncthreads(); });
        __syncthreads();  // shared memory is restaged for the next matrix
        ci = ni;
        cs = ns;
        cU = nU;
        cub = nub;
        cue = nue;
    }
}

// ================================================================== stream kernel (L1 only)
// Shared memory: ring [W*D stages of kKC records] | header (mbarriers, flag) | x in B-fragment
// order | x group sums | chunk partials [tiles_per_pass * cpt][16][B].
template <int W, int D, bool MMA, int BT>
__global__ void __launch_bounds__((W + 1) * 32, 1) q4_stream_kernel(const __grid_constant__ Params p) {
    constexpr int S = W * D;
    static_assert(2 * S * 8 + 4 <= kHdrBytes, "ring header too small");
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * kStageBytes);
    uint64_t* empty = full + S;
    int* flag = reinterpret_cast<int*>(empty + S);
    unsigned char* region = smem + S * kStageBytes + kHdrBytes;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int B = p.B;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        fence_barrier_init();
    }
    __syncthreads();
    allow_dependents();

    if (warp == W) {
        // ---- producer: global chunk c goes to warp c % W, whose r-th chunk (r = c / W) uses stage
        // (c % W) + (r % D) * W in round r / D.  Weights are read-only, so streaming may start
        // before the previous kernel in the stream has finished.
        if (lane == 0) {
            uint32_t c = 0;
            for (int i = 0; i < p.n_mats; ++i) {
                const MatDesc& m = p.m[i];
                Share s;
                if (!cta_share<true>(m, blockIdx.x, s)) continue;
                const int G = m.K >> 7;
                const int cpt = (s.Gs + kKC - 1) / kKC;
                for (int t0 = 0; t0 < s.T; t0 += m.tiles_per_pass) {
                    const int tp = min(m.tiles_per_pass, s.T - t0);
                    for (int lc = 0; lc < tp * cpt; ++lc, ++c) {
                        const int tile = t0 + lc / cpt;
                        const int kc = lc % cpt;
                        const int ng = min(kKC, s.Gs - kc * kKC);
                        const uint32_t r = c / W;
                        const int slot = static_cast<int>(c % W) + static_cast<int>(r % D) * W;
                        const uint32_t round = r / D;
                        if (round > 0 && !mbar_wait(&empty[slot], (round & 1) ^ 1, p.wait_limit)) report_timeout();
                        mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(ng * kRecBytes));
                        const uint8_t* src =
                            m.tiled + (static_cast<size_t>(s.t0 + tile) * G + s.g0 + kc * kKC) * kRecBytes;
                        bulk_g2s(ring + slot * kStageBytes, src, static_cast<uint32_t>(ng * kRecBytes), &full[slot]);
                    }
                }
            }
        }
        return;
    }

    // ---- consumers
    grid_dependency_wait();  // x may be the previous kernel's output; y and ws are shared with it
    constexpr int NT = W * 32;
    const int tid = threadIdx.x;
    const int q = lane >> 2, t = lane & 3;
    uint32_t c = 0;  // global chunk counter, as in the producer
    for (int i = 0; i < p.n_mats; ++i) {
        const MatDesc& m = p.m[i];
        Share s;
        if (!cta_share<true>(m, blockIdx.x, s)) continue;
        const int cpt = (s.Gs + kKC - 1) / kKC;
        uint2* xs = reinterpret_cast<uint2*>(region);
        float* ssum = reinterpret_cast<float*>(region + static_cast<size_t>(s.Gs) * 256 * BT);
        float* fac = ssum + s.Gs * 8;
        unsigned* colmax = reinterpret_cast<unsigned*>(fac + 8);
        float* part = reinterpret_cast<float*>(colmax + 8);
        stage_x_batched<BT, false, false, 1>(m.x, m.K, B, s.g0, s.Gs, xs, ssum, fac, colmax, tid, NT,
                                             [] { consumer_sync<NT>(); });
        consumer_sync<NT>();
        const float f0 = fac[2 * t], f1 = fac[2 * t + 1];
        for (int pass = 0, t0 = 0; t0 < s.T; ++pass, t0 += m.tiles_per_pass) {
            const int tp = min(m.tiles_per_pass, s.T - t0);
            const int prow0 = s.r0 + t0 * 16;
            const int prows = min(tp * 16, s.r1 - prow0);
            const int nch = tp * cpt;
            for (int lc = static_cast<int>((warp + W - c % W) % W); lc < nch; lc += W) {
                const uint32_t cc_g = c + lc;
                const uint32_t r = cc_g / W;
                const int slot = warp + static_cast<int>(r % D) * W;
                if (!mbar_wait(&full[slot], (r / D) & 1, p.wait_limit)) report_timeout();
                const int jj = lc / cpt;
                const int kc = lc - jj * cpt;
                const int ng = min(kKC, s.Gs - kc * kKC);
                const unsigned char* stg = ring + slot * kStageBytes;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                for (int gi = 0; gi < ng; ++gi) {
                    const int gl = kc * kKC + gi;
                    const unsigned char* rec = stg + gi * kRecBytes;
                    const uint4 qa = lds128(rec + 16 * lane);
                    const uint4 qb = lds128(rec + 512 + 16 * lane);
                    const uint2 sc = lds64(rec + 1024 + 8 * q);
                    float cc[4];
                    group_dot<MMA, BT>(qa, qb, xs + xfrag_index<BT>(gl, 0, 0), lane, B, cc);
                    group_epilogue(acc, cc, sc.x, sc.y, ssum + gl * 8 + 2 * t, f0, f1);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);  // release: the reads above are done
                float* pp = part + static_cast<size_t>(lc) * 16 * B;
                const int c0 = 2 * t, c1 = 2 * t + 1;
                if (c0 < B) { pp[q * B + c0] = acc[0]; pp[(q + 8) * B + c0] = acc[2]; }
                if (c1 < B) { pp[q * B + c1] = acc[1]; pp[(q + 8) * B + c1] = acc[3]; }
            }
            c += nch;
            consumer_sync<NT>();
            // add the chunk partials of each row in chunk order
            for (int idx = tid; idx < prows * B; idx += NT) {
                const int b = idx / prows;
                const int rr = idx - b * prows;
                const int jj = rr >> 4, rl = rr & 15;
                float sum = 0.f;
                for (int kc = 0; kc < cpt; ++kc) sum += part[((jj * cpt + kc) * 16 + rl) * B + b];
                store_row_sum(m, s, b, prow0 + rr, B, sum);
            }
            finish_rows<NT>(m, s, pass, prow0, prows, B, tid, flag, [] { consumer_sync<NT>(); });
            consumer_sync<NT>();  // partials, x and flag may be overwritten from here on
        }
    }
}

// ================================================================== activation prep + tile kernel
// q4_xprep_kernel: one CTA per matrix stages its activations once, in global memory, as stage_x_batched
// does in shared memory for the kernels above (layout LM): x in B-fragment order scaled per
// column, the per-group sums of x divided by the column factors, and the column factors.
struct PrepJob {
    const uint16_t* x;
    uint2* xf;
    float* S;
    float* fac;
    int K;
    int pad;
};

struct PrepParams {
    int n;
    int B;
    PrepJob j[kMaxMats];
};

constexpr int kPrepThreads = 1024;

template <int BT, bool X8 = false>
__global__ void __launch_bounds__(kPrepThreads) q4_xprep_kernel(const __grid_constant__ PrepParams p) {
    __shared__ unsigned colmax[8];
    // The tile kernel after this one may start at once: it streams weights (read-only) until its
    // own wait, which returns only when this grid is complete.
    allow_dependents();
    grid_dependency_wait();  // x may be the previous kernel's output
    const PrepJob& j = p.j[blockIdx.x];
    stage_x_batched<BT, true, X8, 8>(j.x, j.K, p.B, 0, j.K >> 7, j.xf, j.S, j.fac, colmax, threadIdx.x,
                                     kPrepThreads, [] { __syncthreads(); });
}

// q4_tiles_ring_kernel: one CTA per SM, persistent over a list of independent matrices, no
// block-wide barrier after the start.  CTA c owns one row block of every matrix (rotated per
// matrix); its tiles, matrix after matrix, form one list that the warps take from a shared
// counter.  A warp computes a whole 16-row tile: all K/128 groups in order, the sum in
// registers, Y written by the warp.  Each warp streams its records through S shared-memory slots
// with cp.async, S-1 records ahead of the one it computes.  The loading side takes the warp's next
// tile as soon as the current one is fully requested, so loading runs on across tile and matrix
// boundaries, and hands the tiles to the computing side through a small per-warp queue.  Exactly
// one commit group per record step (an empty one once the list is exhausted) keeps the wait count
// constant: record c sits in slot c % S, and the slot refilled in step c is the one read in step
// c - 1, whose values are already in registers.  The 64 scale/min bytes are written by lanes 0-3
// and read by all lanes, which cp.async.wait_group + __syncwarp order.  Which warp takes which
// tile changes no arithmetic.
// Inclusive prefix sum of v over threads 0 .. kMaxMats-1 of the block (the other threads pass
// anything; their results are meaningless), and the sum over those threads in *all.  Every thread
// of the block calls it (it holds two block barriers); ws holds kMaxMats / 32 values.
__device__ __forceinline__ int64_t scan_list(int64_t v, int64_t* ws, int64_t* all) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (w >= kMaxMats / 32) v = 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (w < kMaxMats / 32 && lane == 31) ws[w] = v;
    __syncthreads();
    int64_t base = 0, sum = 0;
#pragma unroll
    for (int j = 0; j < kMaxMats / 32; ++j) {
        base += j < w ? ws[j] : 0;
        sum += ws[j];
    }
    *all = sum;
    __syncthreads();  // ws is free for the next call
    return base + v;
}

struct TileMat {
    const uint8_t* tiled;
    const uint4* xf;  // prepared activations, one 16-byte word per lane and fragment pair
    const float* S;   // group sums divided by the column factors
    const float* fac;
    float* y;
    int N, K;
    int row_blocks, rot;
};

struct TileParams {
    int n_mats;
    int B;
    int contiguous;  // 1: CTA c takes a record-balanced contiguous range of the whole tile list
    int pad;
    TileMat m[kMaxMats];
};

constexpr int kItemQ = 16;  // per-warp queue of tiles requested but not yet computed (> S)

// RO: the read-only twin (a measurement aid): the same loads, the same ring, the same tile
// schedule and the same stores, with the unpack, the mma and the scale/min arithmetic replaced by an
// XOR of the loaded words -- the rate this access pattern allows when no arithmetic is done
// (the rumik-oss-1 write-up, "Step 7": a twin of the GEMV that loads but does no maths told
// memory-bound from compute-bound).  Its outputs carry no meaning.
template <int WARPS, int S, int BT, bool RO = false>
__global__ void __launch_bounds__(WARPS * 32, 1) q4_tiles_ring_kernel(const __grid_constant__ TileParams p) {
    static_assert(S >= 2 && S < kItemQ, "ring depth");
    static_assert(WARPS * 32 >= kMaxMats, "one thread per matrix in the prologue");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int prefix[kMaxMats + 1];   // this CTA's tiles in matrices [0, i)
    __shared__ int tfirst[kMaxMats];       // first tile of this CTA's row block in matrix i
    __shared__ int next_item;
    __shared__ int2 itemq[WARPS][kItemQ];  // (matrix, tile)
    __shared__ int64_t scan_ws[kMaxMats / 32];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int t = lane & 3, q = lane >> 2;
    const int B = p.B;
    unsigned char* ring = smem + static_cast<size_t>(warp) * S * kRecBytes;
    const uint32_t ring_s = smem_addr(ring) + 16u * static_cast<uint32_t>(lane);  // this lane's bytes of slot 0
    // This CTA's share of every matrix, thread i for matrix i (in parallel: a serial walk over a
    // long list by one thread costs hundreds of cycles per matrix before any weight is requested),
    // then prefix sums over the matrices by the first kMaxMats threads.
    {
        const int i = threadIdx.x;
        const bool mine = i < p.n_mats;
        const int T_all = mine ? (p.m[i].N + 15) >> 4 : 0;
        const int Gi = mine ? p.m[i].K >> 7 : 1;
        int first = 0, cnt = 0;
        if (p.contiguous) {
            // the list's tiles, matrix after matrix, as one run of records; CTA c takes the tiles
            // whose first record falls in [c R / grid, (c+1) R / grid)
            const int64_t rec = static_cast<int64_t>(T_all) * Gi;
            int64_t R;
            const int64_t cum = scan_list(rec, scan_ws, &R) - rec;
            if (mine) {
                const int64_t nb = gridDim.x, c = blockIdx.x;
                const int64_t lo = c * R / nb, hi = (c + 1) * R / nb;
                // tiles t with cum + t G in [lo, hi)
                int64_t t0 = lo > cum ? (lo - cum + Gi - 1) / Gi : 0;
                int64_t t1 = hi > cum ? (hi - cum + Gi - 1) / Gi : 0;
                t0 = t0 < T_all ? t0 : T_all;
                t1 = t1 < T_all ? t1 : T_all;
                first = static_cast<int>(t0);
                cnt = static_cast<int>(t1 - t0);
            }
        } else if (mine && static_cast<int>(blockIdx.x) < p.m[i].row_blocks) {
            const TileMat& m = p.m[i];
            const int rb = (static_cast<int>(blockIdx.x) + m.rot) % m.row_blocks;
            first = static_cast<int>(static_cast<int64_t>(rb) * T_all / m.row_blocks);
            cnt = static_cast<int>(static_cast<int64_t>(rb + 1) * T_all / m.row_blocks) - first;
        }
        int64_t all;
        const int incl = static_cast<int>(scan_list(static_cast<int64_t>(cnt), scan_ws, &all));
        if (mine) {
            prefix[i] = incl - cnt;
            tfirst[i] = first;
        }
        if (i == 0) {
            prefix[p.n_mats] = static_cast<int>(all);
            next_item = 0;
        }
    }
    __syncthreads();
    const int total = prefix[p.n_mats];

    // ---- loading side (warp-uniform state)
    int scan = 0;  // matrix cursor: items only increase, so it only moves forward
    const uint8_t* ld_ptr = nullptr;
    int ld_left = 0;  // records of the current tile not yet requested
    bool ld_done = false;
    int nq = 0;  // tiles handed to the computing side
    // record r goes to the slot at byte offset (r % S) * kRecBytes
    auto issue = [&](int slot_off) {
        if (ld_left == 0 && !ld_done) {
            int item = 0;
            if (lane == 0) item = atomicAdd(&next_item, 1);
            item = __shfl_sync(0xffffffffu, item, 0);
            if (item < total) {
                while (prefix[scan + 1] <= item) ++scan;
                const TileMat& m = p.m[scan];
                const int G = m.K >> 7;
                const int tile = tfirst[scan] + (item - prefix[scan]);
                ld_ptr = m.tiled + static_cast<size_t>(tile) * G * kRecBytes + 16 * lane;
                ld_left = G;
                if (lane == 0) itemq[warp][nq % kItemQ] = make_int2(scan, tile);
                ++nq;
            } else {
                ld_done = true;
            }
        }
        if (ld_left > 0) {
            const uint32_t dst = ring_s + static_cast<uint32_t>(slot_off);
            cp_async16_s(dst, ld_ptr);
            cp_async16_s(dst + 512, ld_ptr + 512);
            if (lane < 4) cp_async16_s(dst + 1024, ld_ptr + 1024);
            ld_ptr += kRecBytes;
            --ld_left;
        }
        cp_async_commit();
    };
#pragma unroll
    for (int s = 0; s < S - 1; ++s) issue(s * kRecBytes);  // weights are read-only: before the wait

    grid_dependency_wait();  // the prepared activations come from the kernel before
    allow_dependents();

    // ---- computing side
    // Lanes whose batch column is >= B read column 0's activations: the mma keeps batch columns
    // apart, and those outputs are never stored.
    const int xlane = q < B ? lane : t;
    int pq = 0;  // tiles taken from the queue
    int mi = 0, tile = 0, G = 0, g = 0;
    const uint4* xg = nullptr;  // this group's activation words for this lane
    const float* Sg = nullptr;  // this group's sums for columns 2t, 2t+1
    auto take_tile = [&]() {
        __syncwarp();  // lane 0's queue entry is visible to all lanes
        const int2 e = itemq[warp][pq % kItemQ];
        ++pq;
        mi = e.x;
        tile = e.y;
        const TileMat& m = p.m[mi];
        G = m.K >> 7;
        g = 0;
        xg = m.xf + xlane;
        Sg = m.S + 2 * t;
    };
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int rd = 0;                    // slot of this step's record
    int prev = (S - 1) * kRecBytes;  // slot read in the step before (the first step's is unused)
    // one record step; false once the warp's list is done
    auto step = [&]() -> bool {
        cp_async_wait<S - 2>();  // this step's record has landed
        __syncwarp();
        // plain coherent loads: the prepared activations were written by the kernel before, and the
        // grid-dependency wait above them is a compiler barrier for memory accesses
        uint4 xv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) xv[j] = xg[j * (4 * BT)];
        const uint2 sv = *reinterpret_cast<const uint2*>(Sg);
        const uint32_t rec = ring_s + static_cast<uint32_t>(rd);
        const uint4 qa = lds128_s(rec);
        const uint4 qb = lds128_s(rec + 512);
        const uint2 sc = lds64_s(rec - 16u * static_cast<uint32_t>(lane) + 1024u + 8u * static_cast<uint32_t>(q));
        issue(prev);  // S - 1 records ahead, into the slot read one step ago
        prev = rd;
        rd = rd + kRecBytes == S * kRecBytes ? 0 : rd + kRecBytes;
        if constexpr (RO) {
            uint32_t v = qa.x ^ qa.y ^ qa.z ^ qa.w ^ qb.x ^ qb.y ^ qb.z ^ qb.w ^ sc.x ^ sc.y ^ sv.x ^ sv.y;
#pragma unroll
            for (int j = 0; j < 4; ++j) v ^= xv[j].x ^ xv[j].y ^ xv[j].z ^ xv[j].w;
            acc[g & 3] = __uint_as_float(__float_as_uint(acc[g & 3]) ^ v);
            xg += 16 * BT;
            Sg += 8;
        } else {
        float cc[4];
        group_dot_x4(qa, qb, xv, cc);
        const float Sx = __uint_as_float(sv.x), Sy = __uint_as_float(sv.y);
        const float sa = half_bits_to_f32(sc.x), ma = half_bits_to_f32(sc.x >> 16);
        const float sb = half_bits_to_f32(sc.y), mb = half_bits_to_f32(sc.y >> 16);
        acc[0] = fmaf(sa, cc[0], acc[0]);
        acc[0] = fmaf(ma, Sx, acc[0]);
        acc[1] = fmaf(sa, cc[1], acc[1]);
        acc[1] = fmaf(ma, Sy, acc[1]);
        acc[2] = fmaf(sb, cc[2], acc[2]);
        acc[2] = fmaf(mb, Sx, acc[2]);
        acc[3] = fmaf(sb, cc[3], acc[3]);
        acc[3] = fmaf(mb, Sy, acc[3]);
        xg += 16 * BT;
        Sg += 8;
        }
        if (++g < G) return true;
        const TileMat& m = p.m[mi];
        const float f0 = ld_dep_f32(m.fac + 2 * t), f1 = ld_dep_f32(m.fac + 2 * t + 1);
        const int ra = 16 * tile + q, rbw = ra + 8;
        const int c0 = 2 * t, c1 = 2 * t + 1;
        if (ra < m.N) {
            if (c0 < B) m.y[static_cast<size_t>(c0) * m.N + ra] = acc[0] * f0;
            if (c1 < B) m.y[static_cast<size_t>(c1) * m.N + ra] = acc[1] * f1;
        }
        if (rbw < m.N) {
            if (c0 < B) m.y[static_cast<size_t>(c0) * m.N + rbw] = acc[2] * f0;
            if (c1 < B) m.y[static_cast<size_t>(c1) * m.N + rbw] = acc[3] * f1;
        }
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
        // the next tile's first record was requested at least one step ago, so the queue holds it
        // unless the list is exhausted
        if (pq == nq) return false;
        take_tile();
        return true;
    };
    if (nq > 0) {
        take_tile();
#pragma unroll 1
        while (step()) {
        }
    }
    cp_async_wait<0>();
}

// q4_flat_kernel: one matrix per launch, the work split evenly over every warp of the grid.  In the
// tiled layout a matrix is one run of records, tile after tile (G = K/128 records a tile).  CTA c
// takes a contiguous range of whole tiles (the ranges differ by at most one tile), and its WARPS
// warps split the range's records evenly: with R = WARPS u + e records, warp w takes u + 1
// records if w < e, else u, in warp order.  So each warp's share is one contiguous byte range,
// which lane 0 asks L2 for at once (up to kFlatPf records, then kFlatPf ahead of the loads),
// streamed through S shared-memory slots with cp.async as in q4_tiles_ring_kernel.  A warp's
// records split at tile boundaries into segments.  A segment that covers a whole tile writes Y
// directly; the others (at most the first and the last of a warp) leave their partial sums in
// shared memory (slot 0 for the first, slot 1 for the last) and count themselves in the ticket of
// the tile's first warp; the warp that completes the count adds the partials in warp (= record)
// order and writes Y.  Nothing is shared between CTAs and nothing outlives the launch.
// XS: the CTA stages the activations itself (stage_x_batched, layout LM) into shared memory after its
// grid-dependency wait, while its first weight records are already on the way; otherwise they
// come prepared from q4_xprep_kernel in global memory.
// The split depends on N, K and the SM count only, so each batch column is computed in the same
// order for every B.
constexpr int kFlatPf = 16;

struct FlatParams {
    const uint8_t* tiled;
    const uint16_t* x;  // XS: the activations
    const uint4* xf;    // otherwise: prepared activations (layout LM) ...
    const float* S;     // ... group sums divided by the column factors
    const float* fac;   // ... column factors
    float* y;           // may be null (int8 head: only the argmax wanted)
    const uint16_t* rscale;  // int8 head: fp16 scale per row
    int2* cand;         // int8 head, when not null: per CTA and batch column the best (value bits, row)
    int N, K, B;
    int T;   // tiles
    int pf;  // int8 head: records of the run requested into L2 ahead of the loads (int4: kFlatPf)
    int pad;
};

// Argmax order: NaN above every number (lowest index first among NaNs), then larger values, then
// the lower index among equal values (numpy's argmax).  A total order, so any visiting order gives
// the same winner.
__device__ __forceinline__ bool ranks_above(float v, int i, float bv, int bi) {
    const bool vn = v != v, bn = bv != bv;
    if (vn || bn) return vn && (!bn || i < bi);
    return v > bv || (v == bv && i < bi);
}


// ---- int8 head operands (Q8).  An int8 code c becomes the byte c + 128 by flipping its top bit;
// a byte m in the low 8 bits of a bf16 with exponent field 0 or 1 is exactly m * 2^-133 (as for
// the int4 codes), so one LOP3 turns bytes 0 and 2 of a word into an mma operand pair, and a shift
// and a LOP3 bytes 1 and 3.  The offset is removed per record (128-column group g):
// acc += c_g - 128 S_g, so that the running sum keeps the size of the result (summing the
// offset terms over a whole row first makes the tensor-core sums about 80 times larger than
// the result and their rounding visible); y = acc f scale.
__device__ __forceinline__ uint32_t q8_lo(uint32_t w) { return (w & 0x00FF00FFu) ^ 0x00800080u; }
__device__ __forceinline__ uint32_t q8_hi(uint32_t w) { return ((w >> 8) & 0x00FF00FFu) ^ 0x00800080u; }

// c = the record's 16 rows x 8 columns over 128 k of (code + 128) x.  ra/rb: the lane's 32 code
// bytes of rows q and q+8 (k = 32t .. 32t+31 of the group); xv[j]: mma 2j (x, y) and 2j+1 (z, w)
// fragments.
__device__ __forceinline__ void q8_dot(const uint4& ra0, const uint4& ra1, const uint4& rb0, const uint4& rb1,
                                       const uint4 (&xv)[4], float (&c)[4]) {
    const uint32_t wa[8] = {ra0.x, ra0.y, ra0.z, ra0.w, ra1.x, ra1.y, ra1.z, ra1.w};
    const uint32_t wb[8] = {rb0.x, rb0.y, rb0.z, rb0.w, rb1.x, rb1.y, rb1.z, rb1.w};
    float c2[4];  // two chains (mma 0-3 and 4-7), added at the end: a fixed order
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        float (&d)[4] = m < 4 ? c : c2;
        const uint32_t b0 = (m & 1) ? xv[m >> 1].z : xv[m >> 1].x;
        const uint32_t b1 = (m & 1) ? xv[m >> 1].w : xv[m >> 1].y;
        if (m == 0 || m == 4)
            mma_bf16_m16n8k16_zc(d, q8_lo(wa[m]), q8_lo(wb[m]), q8_hi(wa[m]), q8_hi(wb[m]), b0, b1);
        else
            mma_bf16_m16n8k16(d, q8_lo(wa[m]), q8_lo(wb[m]), q8_hi(wa[m]), q8_hi(wb[m]), b0, b1);
    }
    c[0] += c2[0];
    c[1] += c2[1];
    c[2] += c2[2];
    c[3] += c2[3];
}

template <int WARPS, int S, int BT, bool XS, bool Q8 = false>
__global__ void __launch_bounds__(WARPS * 32, 1) q4_flat_kernel(const __grid_constant__ FlatParams p) {
    static_assert(S >= 2, "ring depth");
    constexpr int kRec = Q8 ? kRec8Bytes : kRecBytes;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int ticket[WARPS];
    __shared__ unsigned colmax[8];
    __shared__ int2 wbest[Q8 ? WARPS : 1][8];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int t = lane & 3, q = lane >> 2;
    const int B = p.B;
    const int G = p.K >> 7;
    unsigned char* ring = smem + static_cast<size_t>(warp) * S * kRec;
    float4* part = reinterpret_cast<float4*>(smem + static_cast<size_t>(WARPS) * S * kRec);  // [WARPS][2][32]
    unsigned char* xsm = reinterpret_cast<unsigned char*>(part + WARPS * 2 * 32);
    if (threadIdx.x < WARPS) ticket[threadIdx.x] = 0;

    // this CTA's tiles and this warp's records (local record index within the CTA's range)
    const int nb = static_cast<int>(gridDim.x);
    const int tu = p.T / nb, te = p.T % nb;
    const int c = static_cast<int>(blockIdx.x);
    const int t0 = c * tu + (c < te ? c : te);
    const int Rc = (tu + (c < te ? 1 : 0)) * G;
    const int u = Rc / WARPS, e = Rc % WARPS;
    auto run_start = [&](int v) { return v * u + (v < e ? v : e); };
    auto owner = [&](int r) { return r < e * (u + 1) ? r / (u + 1) : e + (r - e * (u + 1)) / u; };
    const int r0 = run_start(warp);
    const int n = u + (warp < e ? 1 : 0);

    // ---- loading side
    const int lane_off = Q8 ? 32 * lane : 16 * lane;
    const int pf = Q8 ? p.pf : kFlatPf;
    const uint8_t* ld_ptr = p.tiled + (static_cast<size_t>(t0) * G + r0) * kRec + lane_off;
    int ld_left = n;
    if (lane == 0 && n > 0 && pf > 0) prefetch_l2_bulk(ld_ptr, static_cast<uint32_t>(min(n, pf) * kRec));
    const uint32_t ring_s = smem_addr(ring) + static_cast<uint32_t>(lane_off);  // this lane's bytes of slot 0
    auto issue = [&](int slot_off) {
        if (ld_left > 0) {
            if (lane == 0 && pf > 0 && ld_left > pf)
                prefetch_l2_bulk(ld_ptr + static_cast<size_t>(pf) * kRec, kRec);
            const uint32_t dst = ring_s + static_cast<uint32_t>(slot_off);
            if constexpr (Q8) {
                cp_async16_s(dst, ld_ptr);
                cp_async16_s(dst + 16, ld_ptr + 16);
                cp_async16_s(dst + 1024, ld_ptr + 1024);
                cp_async16_s(dst + 1040, ld_ptr + 1040);
            } else {
                cp_async16_s(dst, ld_ptr);
                cp_async16_s(dst + 512, ld_ptr + 512);
                if (lane < 4) cp_async16_s(dst + 1024, ld_ptr + 1024);
            }
            ld_ptr += kRec;
            --ld_left;
        }
        cp_async_commit();
    };
#pragma unroll
    for (int s = 0; s < S - 1; ++s) issue(s * kRec);  // weights are read-only: before the wait

    grid_dependency_wait();  // x (or its prepared copy) comes from the kernel before
    allow_dependents();

    const uint4* xf;
    const float* Sb;
    const float* fac;
    if constexpr (XS) {
        uint2* xs = reinterpret_cast<uint2*>(xsm);
        float* ssum = reinterpret_cast<float*>(xsm + static_cast<size_t>(G) * 256 * BT);
        float* fs = ssum + G * 8;
        stage_x_batched<BT, true, Q8, 2>(p.x, p.K, B, 0, G, xs, ssum, fs, colmax, static_cast<int>(threadIdx.x),
                                         WARPS * 32, [] { __syncthreads(); });
        __syncthreads();
        xf = reinterpret_cast<const uint4*>(xs);
        Sb = ssum;
        fac = fs;
    } else {
        __syncthreads();  // the tickets
        xf = p.xf;
        Sb = p.S;
        fac = p.fac;
    }
    // XS: explicit shared-memory loads; else plain coherent loads of the prepared copy (written by
    // the kernel before: the grid-dependency wait above is a compiler barrier for memory accesses)
    auto ldx4 = [&](const uint4* a) -> uint4 {
        if constexpr (XS) return lds128(reinterpret_cast<const unsigned char*>(a));
        else return *a;
    };
    auto ldx2 = [&](const float* a) -> uint2 {
        if constexpr (XS) return lds64(reinterpret_cast<const unsigned char*>(a));
        else return *reinterpret_cast<const uint2*>(a);
    };
    auto ldf = [&](const float* a) -> float {
        if constexpr (XS) return *a;
        else return ld_dep_f32(a);
    };

    // ---- computing side
    const int xlane = q < B ? lane : t;  // columns >= B read column 0: their outputs are dropped
    const float f0 = ldf(fac + 2 * t), f1 = ldf(fac + 2 * t + 1);
    const int c0 = 2 * t, c1 = 2 * t + 1;
    int tile = r0 / G;  // local tile
    int g = r0 - tile * G;
    int gs = g;  // first group of the current segment
    bool first_seg = true;
    const uint4* xg = xf + xlane + g * (16 * BT);
    const float* Sg = Sb + 2 * t + g * 8;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int rd = 0, prev = (S - 1) * kRec;
    float bv0 = -__int_as_float(0x7f800000), bv1 = bv0;  // Q8 argmax: best of columns c0, c1 so far
    int bi0 = 0x7fffffff, bi1 = 0x7fffffff;

    auto store_y = [&](const float (&a)[4]) {
        const int ra = 16 * (t0 + tile) + q, rbw = ra + 8;
        float v[4];
        if constexpr (Q8) {
            const float sca = ra < p.N ? half_bits_to_f32(ld_nc_u16(p.rscale + ra)) : 0.f;
            const float scb = rbw < p.N ? half_bits_to_f32(ld_nc_u16(p.rscale + rbw)) : 0.f;
            v[0] = (a[0] * f0) * sca;
            v[1] = (a[1] * f1) * sca;
            v[2] = (a[2] * f0) * scb;
            v[3] = (a[3] * f1) * scb;
            if (p.cand) {
                if (ra < p.N) {
                    if (ranks_above(v[0], ra, bv0, bi0)) { bv0 = v[0]; bi0 = ra; }
                    if (ranks_above(v[1], ra, bv1, bi1)) { bv1 = v[1]; bi1 = ra; }
                }
                if (rbw < p.N) {
                    if (ranks_above(v[2], rbw, bv0, bi0)) { bv0 = v[2]; bi0 = rbw; }
                    if (ranks_above(v[3], rbw, bv1, bi1)) { bv1 = v[3]; bi1 = rbw; }
                }
            }
        } else {
            v[0] = a[0] * f0;
            v[1] = a[1] * f1;
            v[2] = a[2] * f0;
            v[3] = a[3] * f1;
        }
        if (p.y == nullptr) return;
        if (ra < p.N) {
            if (c0 < B) p.y[static_cast<size_t>(c0) * p.N + ra] = v[0];
            if (c1 < B) p.y[static_cast<size_t>(c1) * p.N + ra] = v[1];
        }
        if (rbw < p.N) {
            if (c0 < B) p.y[static_cast<size_t>(c0) * p.N + rbw] = v[2];
            if (c1 < B) p.y[static_cast<size_t>(c1) * p.N + rbw] = v[3];
        }
    };
    auto flush = [&](int ge) {  // segment [gs, ge) of `tile` is complete
        if (gs == 0 && ge == G) {
            store_y(acc);
            return;
        }
        part[(warp * 2 + (first_seg ? 0 : 1)) * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        __threadfence_block();
        __syncwarp();
        const int tb = tile * G;
        const int wf = owner(tb), wl = owner(tb + G - 1);  // the warps sharing this tile
        int tk = 0;
        if (lane == 0) tk = atomicAdd(&ticket[wf], 1);
        tk = __shfl_sync(0xffffffffu, tk, 0);
        if (tk != wl - wf) return;
        __threadfence_block();  // every partial of the tile is visible
        // warp wf's segment is its last one (slot 1) when its run began in an earlier tile; every
        // other segment opens its warp's run (slot 0)
        const volatile float4* pp = part + (wf * 2 + (run_start(wf) < tb ? 1 : 0)) * 32 + lane;
        float s[4] = {pp->x, pp->y, pp->z, pp->w};
        for (int v = wf + 1; v <= wl; ++v) {
            pp = part + (v * 2) * 32 + lane;
            s[0] += pp->x;
            s[1] += pp->y;
            s[2] += pp->z;
            s[3] += pp->w;
        }
        store_y(s);
    };

#pragma unroll 1
    for (int i = 0; i < n; ++i) {
        cp_async_wait<S - 2>();  // this step's record has landed
        __syncwarp();
        uint4 xv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) xv[j] = ldx4(xg + j * (4 * BT));
        const uint32_t rec = ring_s + static_cast<uint32_t>(rd);  // this lane's bytes of the record
        if constexpr (Q8) {
            const uint2 sv = ldx2(Sg);
            const uint4 ra0 = lds128_s(rec), ra1 = lds128_s(rec + 16);
            const uint4 rb0 = lds128_s(rec + 1024), rb1 = lds128_s(rec + 1040);
            issue(prev);  // S - 1 records ahead, into the slot read one step ago
            prev = rd;
            rd = rd + kRec == S * kRec ? 0 : rd + kRec;
            float cc[4];
            q8_dot(ra0, ra1, rb0, rb1, xv, cc);
            const float Sx = __uint_as_float(sv.x), Sy = __uint_as_float(sv.y);
            acc[0] += fmaf(-128.f, Sx, cc[0]);
            acc[1] += fmaf(-128.f, Sy, cc[1]);
            acc[2] += fmaf(-128.f, Sx, cc[2]);
            acc[3] += fmaf(-128.f, Sy, cc[3]);
            Sg += 8;
        } else {
            const uint2 sv = ldx2(Sg);
            const uint4 qa = lds128_s(rec);
            const uint4 qb = lds128_s(rec + 512);
            const uint2 sc = lds64_s(rec - static_cast<uint32_t>(lane_off) + 1024u + 8u * static_cast<uint32_t>(q));
            issue(prev);  // S - 1 records ahead, into the slot read one step ago
            prev = rd;
            rd = rd + kRec == S * kRec ? 0 : rd + kRec;
            float cc[4];
            group_dot_x4(qa, qb, xv, cc);
            const float Sx = __uint_as_float(sv.x), Sy = __uint_as_float(sv.y);
            const float sa = half_bits_to_f32(sc.x), ma = half_bits_to_f32(sc.x >> 16);
            const float sb = half_bits_to_f32(sc.y), mb = half_bits_to_f32(sc.y >> 16);
            acc[0] = fmaf(sa, cc[0], acc[0]);
            acc[0] = fmaf(ma, Sx, acc[0]);
            acc[1] = fmaf(sa, cc[1], acc[1]);
            acc[1] = fmaf(ma, Sy, acc[1]);
            acc[2] = fmaf(sb, cc[2], acc[2]);
            acc[2] = fmaf(mb, Sx, acc[2]);
            acc[3] = fmaf(sb, cc[3], acc[3]);
            acc[3] = fmaf(mb, Sy, acc[3]);
            Sg += 8;
        }
        xg += 16 * BT;
        ++g;
        if (g == G || i == n - 1) {
            flush(g);
            first_seg = false;
            acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
            ++tile;
            g = gs = 0;
            xg = xf + xlane;
            Sg = Sb + 2 * t;
        }
    }
    cp_async_wait<0>();
    if constexpr (Q8) {
        if (p.cand) {  // this CTA's best row per batch column (columns >= B are never read)
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {  // lanes with the same t hold the same two columns
                const float ov0 = __shfl_xor_sync(0xffffffffu, bv0, o), ov1 = __shfl_xor_sync(0xffffffffu, bv1, o);
                const int oi0 = __shfl_xor_sync(0xffffffffu, bi0, o), oi1 = __shfl_xor_sync(0xffffffffu, bi1, o);
                if (ranks_above(ov0, oi0, bv0, bi0)) { bv0 = ov0; bi0 = oi0; }
                if (ranks_above(ov1, oi1, bv1, bi1)) { bv1 = ov1; bi1 = oi1; }
            }
            if (q == 0) {
                wbest[warp][c0] = make_int2(__float_as_int(bv0), bi0);
                wbest[warp][c1] = make_int2(__float_as_int(bv1), bi1);
            }
            __syncthreads();
            if (threadIdx.x < 8) {
                float bv = -__int_as_float(0x7f800000);
                int bi = 0x7fffffff;
                for (int w2 = 0; w2 < WARPS; ++w2) {
                    const int2 cv = wbest[w2][threadIdx.x];
                    if (ranks_above(__int_as_float(cv.x), cv.y, bv, bi)) { bv = __int_as_float(cv.x); bi = cv.y; }
                }
                p.cand[blockIdx.x * 8 + threadIdx.x] = make_int2(__float_as_int(bv), bi);
            }
        }
    }
}

// The int8 head's argmax: per batch column the best of the per-CTA candidates of q4_flat_kernel
// ([n_cta][8]).  One CTA of 256 threads: thread t takes candidates t, t + 256, ... (all of column
// t % 8; their loads are independent), then lanes of one column combine by shuffles and the
// warps through shared memory.  ranks_above is a total order, so the combining order is free.
__global__ void __launch_bounds__(256) q8_argmax_final(const int2* cand, int n_cta, int B, int32_t* idx) {
    __shared__ int2 wb[8][8];
    grid_dependency_wait();  // the candidates come from the kernel before
    allow_dependents();      // whatever follows writes only after its own wait
    const int tid = static_cast<int>(threadIdx.x);
    float bv = -__int_as_float(0x7f800000);
    int bi = 0x7fffffff;
    const int n = n_cta * 8;
    uint2 v[5];
#pragma unroll
    for (int u = 0; u < 5; ++u) {  // n <= 5 * 256 for up to 160 CTAs; the rest below
        const int i = tid + u * 256;
        v[u] = i < n ? ld_dep_u2(cand + i) : make_uint2(__float_as_uint(bv), 0x7fffffffu);
    }
#pragma unroll
    for (int u = 0; u < 5; ++u) {
        const float cv = __uint_as_float(v[u].x);
        const int ci = static_cast<int>(v[u].y);
        if (ranks_above(cv, ci, bv, bi)) { bv = cv; bi = ci; }
    }
    for (int i = tid + 5 * 256; i < n; i += 256) {
        const uint2 w = ld_dep_u2(cand + i);
        if (ranks_above(__uint_as_float(w.x), static_cast<int>(w.y), bv, bi)) {
            bv = __uint_as_float(w.x);
            bi = static_cast<int>(w.y);
        }
    }
#pragma unroll
    for (int o = 8; o < 32; o <<= 1) {  // lanes with the same lane % 8 hold the same column
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ranks_above(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    const int lane = tid & 31, warp = tid >> 5;
    if (lane < 8) wb[warp][lane] = make_int2(__float_as_int(bv), bi);
    __syncthreads();
    if (tid < B) {
        bv = __int_as_float(wb[0][tid].x);
        bi = wb[0][tid].y;
        for (int w = 1; w < 8; ++w)
            if (ranks_above(__int_as_float(wb[w][tid].x), wb[w][tid].y, bv, bi)) {
                bv = __int_as_float(wb[w][tid].x);
                bi = wb[w][tid].y;
            }
        idx[tid] = bi == 0x7fffffff ? 0 : bi;
    }
}

// ================================================================== argmax

__device__ __forceinline__ float4 ld_dep_f4(const float4* p) {
    float4 r;
    asm volatile("ld.global.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "l"(p)
                 : "memory");
    return r;
}

// One CTA per row.  The row is read as 16-byte words, four independent loads in flight per
// thread (a scalar head up to the first 16-byte boundary and a scalar tail); ranks_above is a
// total order, so the visiting order does not change the result.
__global__ void __launch_bounds__(1024) q4_argmax_kernel(const float* __restrict__ Y, int N, int32_t* idx) {
    grid_dependency_wait();  // Y is usually the previous kernel's output
    const float* row = Y + static_cast<size_t>(blockIdx.x) * N;
    float bv = -__int_as_float(0x7f800000);
    int bi = 0x7fffffff;
    auto consider = [&](float v, int i) {
        if (ranks_above(v, i, bv, bi)) { bv = v; bi = i; }
    };
    const int mis = static_cast<int>((reinterpret_cast<uintptr_t>(row) & 15u) >> 2);  // row is 4-byte aligned
    const int head = min(N, (4 - mis) & 3);
    const int n4 = (N - head) >> 2;
    const int tail0 = head + 4 * n4;
    const int tid = static_cast<int>(threadIdx.x);
    if (tid < head) consider(ld_dep_f32(row + tid), tid);
    if (tail0 + tid < N) consider(ld_dep_f32(row + tail0 + tid), tail0 + tid);
    const float4* row4 = reinterpret_cast<const float4*>(row + head);
    constexpr int kU = 4;
    for (int base = tid; base < n4; base += kU * 1024) {
        float4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int j = base + u * 1024;
            v[u] = j < n4 ? ld_dep_f4(row4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int j = base + u * 1024;
            if (j < n4) {
                const int i = head + 4 * j;
                consider(v[u].x, i);
                consider(v[u].y, i + 1);
                consider(v[u].z, i + 2);
                consider(v[u].w, i + 3);
            }
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ranks_above(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    __shared__ float sv[32];
    __shared__ int si[32];
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) { sv[w] = bv; si[w] = bi; }
    __syncthreads();
    if (w == 0) {
        const int nw = blockDim.x >> 5;
        bv = (threadIdx.x < nw) ? sv[threadIdx.x] : -__int_as_float(0x7f800000);
        bi = (threadIdx.x < nw) ? si[threadIdx.x] : 0x7fffffff;
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ranks_above(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if (threadIdx.x == 0) idx[blockIdx.x] = (bi == 0x7fffffff) ? 0 : bi;
    }
}

// ================================================================== top-k Gumbel-max sampler
// q4_sample_kernel: one CTA of 1024 threads per batch row of logits.  The top k follow the argmax
// order (NaN above every number, larger first, lower index first among equal values): a 32-bit
// key that grows with that order (rank_key) and, packed with the complemented index below it, a
// 64-bit key that is unique and sorts the same way.  (1) Each thread keeps the 4 best keys of its
// elements; the k-th best of those 4096 (a radix select in shared memory), tau, has at least k
// elements at or above it, so the top k all lie at or above tau.  Every element >= tau is gathered
// (one ballot per warp step) and, when they fit in kSampleCap, sorted by their 64-bit keys
// (bitonic, descending) -- the first k are the ranked top k.  When they do not fit (long runs of
// equal values), a radix select over the key's four bytes, most significant first, finds the k-th
// best key T instead: elements above T all belong to the top k, and of those equal to T the
// lowest-index ones fill the rest; those k are gathered and sorted.
// (3) Thread r scores rank r as fp32(fp32(y * inv_temperature) + noise[r]) -- two rounded
// operations, never fused -- and the best score (NaN first, ties to the lower rank) picks the token.
constexpr int kSampleThreads = 1024;
constexpr int kSampleMaxK = 1024;
constexpr int kSampleCap = 2048;  // candidates held in shared memory (>= kSampleMaxK)

__device__ __forceinline__ uint32_t rank_key(float v) {
    if (v != v) return 0xFFFFFFFFu;  // NaN: above every number
    uint32_t b = __float_as_uint(v);
    if ((b & 0x7FFFFFFFu) == 0) b = 0;  // -0 and +0 are equal values
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// ================================================================== argmax keys (row-sharded heads)
// The best logit of a row slice as one 64-bit key that orders like the argmax rule over the whole
// row: bits 63..32 the value's rank_key, bits 31..0 the complement of its global index (a lower
// index ranks higher among equal values).  Stored with the top bit flipped, so that signed 64-bit
// order -- what a MAX all-reduce of int64 compares -- equals that unsigned order.  The best key of
// several slices is the largest; its low 32 bits, complemented, are the global index.
__device__ __forceinline__ uint64_t argmax_key(float v, uint32_t gidx) {
    return (static_cast<uint64_t>(rank_key(v)) << 32) | static_cast<uint64_t>(~gidx);
}

// One CTA per row, the row read as in q4_argmax_kernel (16-byte words, scalar head and tail); the
// largest key wins, so the visiting order does not matter.
__global__ void __launch_bounds__(1024) q4_argmax_key_kernel(const float* __restrict__ Y, int N, uint32_t base,
                                                             int64_t* keys) {
    grid_dependency_wait();
    const float* row = Y + static_cast<size_t>(blockIdx.x) * N;
    uint64_t best = 0;
    auto consider = [&](float v, int i) {
        const uint64_t k = argmax_key(v, base + static_cast<uint32_t>(i));
        best = k > best ? k : best;
    };
    const int mis = static_cast<int>((reinterpret_cast<uintptr_t>(row) & 15u) >> 2);
    const int head = min(N, (4 - mis) & 3);
    const int n4 = (N - head) >> 2;
    const int tail0 = head + 4 * n4;
    const int tid = static_cast<int>(threadIdx.x);
    if (tid < head) consider(ld_dep_f32(row + tid), tid);
    if (tail0 + tid < N) consider(ld_dep_f32(row + tail0 + tid), tail0 + tid);
    const float4* row4 = reinterpret_cast<const float4*>(row + head);
    for (int j = tid; j < n4; j += 1024) {
        const float4 v = ld_dep_f4(row4 + j);
        const int i = head + 4 * j;
        consider(v.x, i);
        consider(v.y, i + 1);
        consider(v.z, i + 2);
        consider(v.w, i + 3);
    }
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t ok = __shfl_xor_sync(0xffffffffu, best, o);
        best = ok > best ? ok : best;
    }
    __shared__ uint64_t sk[32];
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) sk[w] = best;
    __syncthreads();
    if (w == 0) {
        best = threadIdx.x < (blockDim.x >> 5) ? sk[threadIdx.x] : 0;
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t ok = __shfl_xor_sync(0xffffffffu, best, o);
            best = ok > best ? ok : best;
        }
        if (threadIdx.x == 0) keys[blockIdx.x] = static_cast<int64_t>(best ^ 0x8000000000000000ull);
    }
}

__global__ void q4_argmax_key_index_kernel(const int64_t* __restrict__ keys, int B, int32_t* idx) {
    grid_dependency_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) idx[b] = static_cast<int32_t>(~static_cast<uint32_t>(static_cast<uint64_t>(keys[b])));
}

template <bool VEC>
__global__ void __launch_bounds__(kSampleThreads) q4_sample_kernel(const float* Y, int N, int k, float inv_t,
                                                                   const float* noise, int32_t* token,
                                                                   int32_t* topk) {
    __shared__ unsigned hist[256];
    __shared__ uint32_t sample[4 * kSampleThreads];
    __shared__ unsigned long long cand[kSampleCap];
    __shared__ unsigned sh_prefix, sh_remain, sh_ties, sh_count, sh_tie_base;
    __shared__ unsigned warp_sum[32];
    __shared__ float best_s[32];
    __shared__ int best_r[32];
    grid_dependency_wait();  // the logits are usually the previous kernel's output
    allow_dependents();
    const int tid = static_cast<int>(threadIdx.x);
    const int lane = tid & 31, warp = tid >> 5;
    const float* row = Y + static_cast<size_t>(blockIdx.x) * N;
    constexpr int U = 8;  // loads in flight per thread
    auto key_at = [&](int i) -> uint32_t { return rank_key(ld_dep_f32(row + i)); };
    // fn(index, value) over the whole row: VEC reads 16-byte words (row 16-byte aligned, N % 4 == 0),
    // U independent loads in flight per thread, coalesced across the block
    auto for_row = [&](auto&& fn) {
        if constexpr (VEC) {
            const float4* row4 = reinterpret_cast<const float4*>(row);
            const int n4 = N >> 2;
            for (int base = tid; base < n4; base += U * kSampleThreads) {
                float4 v[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int j = base + u * kSampleThreads;
                    v[u] = j < n4 ? ld_dep_f4(row4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int j = base + u * kSampleThreads;
                    if (j < n4) {
                        fn(4 * j, v[u].x);
                        fn(4 * j + 1, v[u].y);
                        fn(4 * j + 2, v[u].z);
                        fn(4 * j + 3, v[u].w);
                    }
                }
            }
        } else {
            for (int base = tid; base < N; base += U * kSampleThreads) {
                float v[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = base + u * kSampleThreads;
                    v[u] = i < N ? ld_dep_f32(row + i) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = base + u * kSampleThreads;
                    if (i < N) fn(i, v[u]);
                }
            }
        }
    };

    // bitonic sort, descending, of a[0..P) (P a power of two) by the whole block
    auto sort_desc = [&](auto* a, int P) {
        for (int size = 2; size <= P; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int i = tid; i < P; i += kSampleThreads) {
                    const int j = i ^ stride;
                    if (j > i) {
                        const bool desc = (i & size) == 0;  // descending runs where the size bit is clear
                        const auto x = a[i], y = a[j];
                        if (desc ? (x < y) : (x > y)) {
                            a[i] = y;
                            a[j] = x;
                        }
                    }
                }
                __syncthreads();
            }
        }
    };
    auto pack = [](uint32_t key, int i) {
        return (static_cast<unsigned long long>(key) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(i));
    };
    // warp 0: the digit d whose bin holds the remain-th largest counted key, scanning bins from 255
    // down; lane l holds bins 255-8l .. 248-8l, a shuffle scan finds the crossing lane.  Writes
    // sh_prefix (prefix | d << shift), sh_remain (remain minus the keys in higher bins), sh_ties.
    auto select_digit = [&](uint32_t prefix, int shift, unsigned remain) {
        if (warp != 0) return;
        unsigned c[8], local = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            c[j] = hist[255 - 8 * lane - j];
            local += c[j];
        }
        unsigned incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const unsigned excl = incl - local;
        if (excl < remain && remain <= incl) {
            unsigned above = excl;
            int j = 0;
            for (; j < 7; ++j) {
                if (above + c[j] >= remain) break;
                above += c[j];
            }
            const int d = 255 - 8 * lane - j;
            sh_prefix = prefix | (static_cast<uint32_t>(d) << shift);
            sh_remain = remain - above;
            sh_ties = c[j];
        }
    };

    // (1) the 4 best keys of each thread's elements (0 sorts below every element's key)
    {
        uint32_t t4[4] = {0u, 0u, 0u, 0u};
        for_row([&](int, float v) {
            const uint32_t key = rank_key(v);
            if (key > t4[3]) {
                if (key > t4[0]) { t4[3] = t4[2]; t4[2] = t4[1]; t4[1] = t4[0]; t4[0] = key; }
                else if (key > t4[1]) { t4[3] = t4[2]; t4[2] = t4[1]; t4[1] = key; }
                else if (key > t4[2]) { t4[3] = t4[2]; t4[2] = key; }
                else t4[3] = key;
            }
        });
#pragma unroll
        for (int m = 0; m < 4; ++m) sample[4 * tid + m] = t4[m];
        if (tid == 0) sh_count = 0;
        __syncthreads();
    }
    // tau = the k-th largest of the 4096 sampled keys: a radix select over them in shared memory
    uint32_t tau;
    {
        uint32_t prefix = 0, mask = 0;
        unsigned remain = static_cast<unsigned>(k);
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            if (tid < 256) hist[tid] = 0;
            __syncthreads();
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t key = sample[m * kSampleThreads + tid];
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
            }
            __syncthreads();
            select_digit(prefix, shift, remain);
            __syncthreads();
            prefix = sh_prefix;
            remain = sh_remain;
            mask |= 0xFFu << shift;
        }
        tau = prefix;
    }
    // gather every element at or above tau: one ballot and one shared counter step per warp step
    for_row([&](int i, float v) {
        const uint32_t key = rank_key(v);
        const bool take = key >= tau;
        const unsigned act = __activemask();
        const unsigned bal = __ballot_sync(act, take);
        const int leader = __ffs(act) - 1;
        unsigned base = 0;
        if (lane == leader && bal) base = atomicAdd(&sh_count, static_cast<unsigned>(__popc(bal)));
        base = __shfl_sync(act, base, leader);
        if (take) {
            const unsigned pos = base + __popc(bal & ((1u << lane) - 1u));
            if (pos < static_cast<unsigned>(kSampleCap)) cand[pos] = pack(key, i);
        }
    });
    __syncthreads();
    int n_cand = static_cast<int>(sh_count);
    if (n_cand > kSampleCap) {  // too many to hold: radix select for the exact k-th best key
        uint32_t prefix = 0, mask = 0;
        unsigned remain = static_cast<unsigned>(k);
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            if (tid < 256) hist[tid] = 0;
            __syncthreads();
            for_row([&](int, float v) {
                const uint32_t key = rank_key(v);
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
            });
            __syncthreads();
            select_digit(prefix, shift, remain);
            __syncthreads();
            prefix = sh_prefix;
            remain = sh_remain;
            mask |= 0xFFu << shift;
        }
        const uint32_t T = prefix;
        const unsigned take_ties = remain;           // elements equal to T to take (>= 1)
        const unsigned above_T = static_cast<unsigned>(k) - take_ties;
        const bool all_ties = sh_ties == take_ties;  // (sh_ties: elements equal to T)

        // (2) gather: keys above T anywhere in [0, above_T); ties in [above_T, k), lowest index first
        if (tid == 0) { sh_count = 0; sh_tie_base = 0; }
        __syncthreads();
        for_row([&](int i, float v) {
            const uint32_t key = rank_key(v);
            const unsigned long long packed =
                (static_cast<unsigned long long>(key) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(i));
            if (key > T) cand[atomicAdd(&sh_count, 1u)] = packed;
            else if (key == T && all_ties) cand[above_T + atomicAdd(&sh_tie_base, 1u)] = packed;
        });
        if (!all_ties) {
            // more elements equal T than needed: walk the row in index order, 1024 at a time, and give
            // each tie its rank among ties by a block-wide exclusive scan
            __syncthreads();
            unsigned running = 0;
            for (int base = 0; base < N && running < take_ties; base += kSampleThreads) {
                const int i = base + tid;
                const unsigned flag = (i < N && key_at(i) == T) ? 1u : 0u;
                const unsigned bal = __ballot_sync(0xffffffffu, flag);
                if (lane == 0) warp_sum[warp] = __popc(bal);
                __syncthreads();
                unsigned before = 0, total = 0;
                for (int w = 0; w < 32; ++w) {
                    const unsigned c = warp_sum[w];
                    if (w < warp) before += c;
                    total += c;
                }
                const unsigned rank = running + before + __popc(bal & ((1u << lane) - 1u));
                if (flag && rank < take_ties)
                    cand[above_T + rank] =
                        (static_cast<unsigned long long>(T) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(i));
                running += total;
                __syncthreads();
            }
        }
        __syncthreads();
        n_cand = k;
    }
    // pad to a power of two with the smallest key and sort descending: the first k are the top k
    int P = 1;
    while (P < n_cand) P <<= 1;
    for (int i = n_cand + tid; i < P; i += kSampleThreads) cand[i] = 0ull;
    __syncthreads();
    sort_desc(cand, P);

    // (3) scores and the token
    float s = -__int_as_float(0x7f800000);
    int r = 0x7fffffff;
    int my_idx = 0;
    if (tid < k) {
        my_idx = static_cast<int>(~static_cast<uint32_t>(cand[tid] & 0xFFFFFFFFull));
        if (topk) topk[static_cast<size_t>(blockIdx.x) * k + tid] = my_idx;
        const float v = ld_dep_f32(row + my_idx);
        s = __fadd_rn(__fmul_rn(v, inv_t), ld_dep_f32(noise + static_cast<size_t>(blockIdx.x) * k + tid));
        r = tid;
    }
    for (int o = 16; o > 0; o >>= 1) {
        const float os = __shfl_xor_sync(0xffffffffu, s, o);
        const int orr = __shfl_xor_sync(0xffffffffu, r, o);
        if (ranks_above(os, orr, s, r)) { s = os; r = orr; }
    }
    if (lane == 0) { best_s[warp] = s; best_r[warp] = r; }
    __syncthreads();
    if (warp == 0) {
        s = best_s[lane];
        r = best_r[lane];
        for (int o = 16; o > 0; o >>= 1) {
            const float os = __shfl_xor_sync(0xffffffffu, s, o);
            const int orr = __shfl_xor_sync(0xffffffffu, r, o);
            if (ranks_above(os, orr, s, r)) { s = os; r = orr; }
        }
        if (lane == 0)
            token[blockIdx.x] = static_cast<int32_t>(~static_cast<uint32_t>(cand[r] & 0xFFFFFFFFull));
    }
}

// ================================================================== top-k sampling over a CTA cluster
// q4_sample_cluster_kernel: the same result as q4_sample_kernel for k <= kClusterMaxK, with each
// row split over a cluster of kSC CTAs on kSC SMs (one row per cluster, grid (kSC, B)).
// (1) CTA c takes chunk c of the row (ceil(N / kSC) rounded up to 4 elements) and finds its own
// top min(k, chunk) by the argmax order, exactly.  Each thread's best key is a sample; a two-pass
// radix select over the top 16 bits of those samples gives L, a lower bound of the chunk's k-th
// best key (the samples are chunk elements, so at least k elements reach it).  Every element at
// or above L is gathered (a count per thread, one scan and one shared atomic per warp) and the
// gathered 64-bit (key, ~index) keys are ranked -- by counting when few, by a bitonic sort
// otherwise.  When more than kSCCap elements reach L (long runs of equal values), an exact radix
// select over the chunk finds the k-th best key T and its ties are taken lowest index first, as
// in q4_sample_kernel.  The CTA writes its sorted list into the leader CTA's shared memory
// (distributed shared memory of this GPU's own SMs), padded with zero keys.
// (2) One cluster barrier; the other CTAs leave.  The leader ranks each entry among all lists (its
// place in its own list plus, in every other list, the number of larger keys, by binary search):
// the entries ranked below k are the row's top k, each scored where it is ranked.
// (3) Scores and the token as in q4_sample_kernel; the logit comes back from its key.
// The row's top k is the union's top k because every element of it is in its own chunk's top k;
// the 64-bit keys are unique, so every rank is.  No wait in this kernel spins: the cluster
// barrier is a hardware barrier that every thread of every CTA of the cluster reaches on every
// path.
constexpr int kSC = 8;             // CTAs per row: one portable-size cluster
constexpr int kSCThreads = 1024;
constexpr int kClusterMaxK = 128;  // larger k uses q4_sample_kernel
constexpr int kSCCap = 2048;       // gathered chunk candidates held in shared memory
constexpr int kSCRegs = 8;         // keys per thread held in registers when the chunk fits
constexpr int kListStride = kClusterMaxK + 1;  // lists one 8-byte word apart in bank order

__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 64-bit store into the shared memory of CTA `rank` of this cluster, at the offset `local` has here
__device__ __forceinline__ void st_cluster_u64(void* local, unsigned rank, unsigned long long v) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(ra), "l"(v) : "memory");
}

// q4_argmax_cluster_kernel: the q4_argmax_kernel result with each row split over a cluster of kAC
// CTAs, so that every thread issues its few 16-byte loads at once (one memory round trip for a
// 65,536-wide row instead of four).  CTA r of a row's cluster takes words [r n4 / kAC, (r+1) n4 / kAC)
// of the row's 16-byte-aligned body (CTA 0 also the scalar head, the last CTA the scalar tail),
// reduces them like q4_argmax_kernel and stores its best (value bits, index) into the shared memory
// of CTA 0; after one cluster barrier CTA 0 merges the kAC candidates.  ranks_above is a total
// order, so the split changes no result.
constexpr int kAC = 8;  // CTAs per row: one portable-size cluster
constexpr int kACThreads = 512;

__global__ void __launch_bounds__(kACThreads) q4_argmax_cluster_kernel(const float* __restrict__ Y, int N,
                                                                       int32_t* idx) {
    __shared__ unsigned long long cand[kAC];  // CTA 0: every CTA's best
    __shared__ float sv[kACThreads / 32];
    __shared__ int si[kACThreads / 32];
    grid_dependency_wait();  // the logits are usually the previous kernel's output
    allow_dependents();
    const int rank = static_cast<int>(blockIdx.x);  // the cluster spans the grid's x dimension (kAC)
    const float* row = Y + static_cast<size_t>(blockIdx.y) * N;
    float bv = -__int_as_float(0x7f800000);
    int bi = 0x7fffffff;
    auto consider = [&](float v, int i) {
        if (ranks_above(v, i, bv, bi)) { bv = v; bi = i; }
    };
    const int mis = static_cast<int>((reinterpret_cast<uintptr_t>(row) & 15u) >> 2);  // row is 4-byte aligned
    const int head = min(N, (4 - mis) & 3);
    const int n4 = (N - head) >> 2;
    const int tail0 = head + 4 * n4;
    const int tid = static_cast<int>(threadIdx.x);
    if (rank == 0 && tid < head) consider(ld_dep_f32(row + tid), tid);
    if (rank == kAC - 1 && tail0 + tid < N) consider(ld_dep_f32(row + tail0 + tid), tail0 + tid);
    const int w0 = static_cast<int>(static_cast<int64_t>(n4) * rank / kAC);
    const int w1 = static_cast<int>(static_cast<int64_t>(n4) * (rank + 1) / kAC);
    const float4* row4 = reinterpret_cast<const float4*>(row + head);
    constexpr int kU = 4;
    for (int base = w0 + tid; base < w1; base += kU * kACThreads) {
        float4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int j = base + u * kACThreads;
            v[u] = j < w1 ? ld_dep_f4(row4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int j = base + u * kACThreads;
            if (j < w1) {
                const int i = head + 4 * j;
                consider(v[u].x, i);
                consider(v[u].y, i + 1);
                consider(v[u].z, i + 2);
                consider(v[u].w, i + 3);
            }
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ranks_above(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    const int w = tid >> 5;
    if ((tid & 31) == 0) { sv[w] = bv; si[w] = bi; }
    __syncthreads();
    if (w == 0) {
        bv = tid < kACThreads / 32 ? sv[tid] : -__int_as_float(0x7f800000);
        bi = tid < kACThreads / 32 ? si[tid] : 0x7fffffff;
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ranks_above(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if (tid == 0)
            st_cluster_u64(&cand[rank], 0u,
                           (static_cast<unsigned long long>(__float_as_uint(bv)) << 32) | static_cast<uint32_t>(bi));
    }
    cluster_barrier();  // every thread of every CTA of the cluster reaches it
    if (rank == 0 && tid == 0) {
        bv = -__int_as_float(0x7f800000);
        bi = 0x7fffffff;
        for (int c = 0; c < kAC; ++c) {
            const float v = __uint_as_float(static_cast<uint32_t>(cand[c] >> 32));
            const int i = static_cast<int>(static_cast<uint32_t>(cand[c]));
            if (ranks_above(v, i, bv, bi)) { bv = v; bi = i; }
        }
        idx[blockIdx.y] = bi == 0x7fffffff ? 0 : bi;
    }
}

// VEC: 16-byte loads (row 16-byte aligned, N a multiple of 4); REG: the chunk's keys fit in
// registers (kSCThreads * kSCRegs) and the row is read once
template <bool VEC, bool REG>
__global__ void __launch_bounds__(kSCThreads) q4_sample_cluster_kernel(const float* Y, int N, int k, float inv_t,
                                                                       const float* noise, int32_t* token,
                                                                       int32_t* topk) {
    __shared__ unsigned hist[2][256];
    __shared__ unsigned long long cand[kSCCap];
    __shared__ unsigned long long all[kSC * kListStride];  // every CTA's list, list c at c * kListStride
    __shared__ float s_noise[kClusterMaxK];
    __shared__ unsigned sh_prefix, sh_remain, sh_ties, sh_count, sh_tie_base;
    __shared__ unsigned warp_sum[kSCThreads / 32];
    __shared__ unsigned long long my_best;            // this CTA's best (score, rank) key
    __shared__ int my_idx[kClusterMaxK];              // this CTA's row index of each of its ranks
    __shared__ unsigned long long cl_best[kSC];       // leader: every CTA's best key
    __shared__ unsigned long long cl_idx[kSC];        // leader: the row index of each CTA's best
    grid_dependency_wait();  // the logits are usually the previous kernel's output
    allow_dependents();
    const int tid = static_cast<int>(threadIdx.x);
    const int lane = tid & 31, warp = tid >> 5;
    const unsigned crank = blockIdx.x;  // the cluster is the kSC CTAs of one blockIdx.y
    const int b = static_cast<int>(blockIdx.y);
    const float* row = Y + static_cast<size_t>(b) * N;
    const int chunk = static_cast<int>(((static_cast<long long>(N) + kSC - 1) / kSC + 3) & ~3LL);
    auto chunk_lo = [&](int c) {
        const long long v = static_cast<long long>(c) * chunk;
        return static_cast<int>(v < N ? v : N);
    };
    const int lo = chunk_lo(static_cast<int>(crank));
    const int len = chunk_lo(static_cast<int>(crank) + 1) - lo;  // the last chunk ends at N
    const int kc = k < len ? k : len;
    const int n4 = len >> 2;
    if (tid < k) s_noise[tid] = ld_dep_f32(noise + static_cast<size_t>(b) * k + tid);
    if (tid < 512) (&hist[0][0])[tid] = 0u;
    if (tid == 0) {
        sh_count = 0u;
        my_best = 0ull;  // below every (score, rank) key
    }
    uint32_t rk[REG ? kSCRegs : 1];  // REG: the keys of this thread's elements (0 where none)
    if constexpr (REG) {
        if constexpr (VEC) {
            const float4* c4 = reinterpret_cast<const float4*>(row + lo);
#pragma unroll
            for (int u = 0; u < kSCRegs / 4; ++u) {
                const int j = tid + u * kSCThreads;
                const float4 x = j < n4 ? ld_dep_f4(c4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                rk[4 * u] = j < n4 ? rank_key(x.x) : 0u;
                rk[4 * u + 1] = j < n4 ? rank_key(x.y) : 0u;
                rk[4 * u + 2] = j < n4 ? rank_key(x.z) : 0u;
                rk[4 * u + 3] = j < n4 ? rank_key(x.w) : 0u;
            }
        } else {
#pragma unroll
            for (int u = 0; u < kSCRegs; ++u) {
                const int i = tid + u * kSCThreads;
                rk[u] = i < len ? rank_key(ld_dep_f32(row + lo + i)) : 0u;
            }
        }
    }
    constexpr int U = 4;
    // fn(index, key) over this CTA's chunk
    auto for_keys = [&](auto&& fn) {
        if constexpr (REG) {
#pragma unroll
            for (int u = 0; u < kSCRegs; ++u) {
                if constexpr (VEC) {
                    const int j = tid + (u >> 2) * kSCThreads;
                    if (j < n4) fn(lo + 4 * j + (u & 3), rk[u]);
                } else {
                    const int i = tid + u * kSCThreads;
                    if (i < len) fn(lo + i, rk[u]);
                }
            }
        } else if constexpr (VEC) {
            const float4* c4 = reinterpret_cast<const float4*>(row + lo);
            for (int base = tid; base < n4; base += U * kSCThreads) {
                float4 v[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int j = base + u * kSCThreads;
                    v[u] = j < n4 ? ld_dep_f4(c4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int j = base + u * kSCThreads;
                    if (j < n4) {
                        fn(lo + 4 * j, rank_key(v[u].x));
                        fn(lo + 4 * j + 1, rank_key(v[u].y));
                        fn(lo + 4 * j + 2, rank_key(v[u].z));
                        fn(lo + 4 * j + 3, rank_key(v[u].w));
                    }
                }
            }
        } else {
            for (int base = tid; base < len; base += U * kSCThreads) {
                float v[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = base + u * kSCThreads;
                    v[u] = i < len ? ld_dep_f32(row + lo + i) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = base + u * kSCThreads;
                    if (i < len) fn(lo + i, rank_key(v[u]));
                }
            }
        }
    };
    auto pack = [](uint32_t key, int i) {
        return (static_cast<unsigned long long>(key) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(i));
    };
    // warp 0: the digit whose bin of h holds the remain-th largest counted key, bins scanned from
    // 255 down (lane l holds bins 255-8l .. 248-8l); writes sh_prefix (prefix | digit << shift),
    // sh_remain (remain minus the keys in higher bins) and sh_ties (the keys in that bin)
    auto select_digit = [&](const unsigned* h, uint32_t prefix, int shift, unsigned remain) {
        if (warp != 0) return;
        unsigned c[8], local = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            c[j] = h[255 - 8 * lane - j];
            local += c[j];
        }
        unsigned incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const unsigned excl = incl - local;
        if (excl < remain && remain <= incl) {
            unsigned above = excl;
            int j = 0;
            for (; j < 7; ++j) {
                if (above + c[j] >= remain) break;
                above += c[j];
            }
            sh_prefix = prefix | (static_cast<uint32_t>(255 - 8 * lane - j) << shift);
            sh_remain = remain - above;
            sh_ties = c[j];
        }
    };
    // bitonic sort, descending, of a[0..P) (P a power of two) by the whole block
    auto sort_desc = [&](unsigned long long* a, int P) {
        for (int size = 2; size <= P; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int i = tid; i < P; i += kSCThreads) {
                    const int j = i ^ stride;
                    if (j > i) {
                        const bool desc = (i & size) == 0;
                        const unsigned long long x = a[i], y = a[j];
                        if (desc ? (x < y) : (x > y)) {
                            a[i] = y;
                            a[j] = x;
                        }
                    }
                }
                __syncthreads();
            }
        }
    };
    // this CTA's list goes to slots crank * kListStride .. of every CTA's `all`
    unsigned long long* my_slots = all + crank * kListStride;
    auto put = [&](int slot, unsigned long long v) {
#pragma unroll
        for (unsigned d = 0; d < kSC; ++d) {
            if (d == crank) my_slots[slot] = v;
            else st_cluster_u64(my_slots + slot, d, v);
        }
    };

    // ---- (1) this chunk's top kc, best first, into the leader's shared memory
    // Shared memory of another CTA may be written only once that CTA runs: the arrive here and the
    // wait before the first such store let the cluster's start-up overlap the selection.
    asm volatile("barrier.cluster.arrive.aligned;" ::: "memory");
    int M = 0;
    if (kc > 0) {
        uint32_t t0 = 0u;  // the thread's best key: its sample
        for_keys([&](int, uint32_t key) { t0 = key > t0 ? key : t0; });
        __syncthreads();  // histograms zeroed
        atomicAdd(&hist[0][t0 >> 24], 1u);
        __syncthreads();
        select_digit(hist[0], 0u, 24, static_cast<unsigned>(kc));
        __syncthreads();
        if ((t0 >> 24) == (sh_prefix >> 24)) atomicAdd(&hist[1][(t0 >> 16) & 255u], 1u);
        __syncthreads();
        select_digit(hist[1], sh_prefix, 16, sh_remain);
        __syncthreads();
        // L: the top 16 bits of the kc-th best sample, a lower bound of the chunk's kc-th best key
        const uint32_t L = sh_prefix;
        if constexpr (REG) {
            // this thread's elements at or above L; one warp scan and one shared atomic per warp
            unsigned mine = 0;
            for_keys([&](int, uint32_t key) { mine += key >= L ? 1u : 0u; });
            if (__any_sync(0xffffffffu, mine != 0)) {
                unsigned incl = mine;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                unsigned base = 0;
                if (lane == 31) base = atomicAdd(&sh_count, incl);
                unsigned pos = __shfl_sync(0xffffffffu, base, 31) + incl - mine;
                if (mine)
                    for_keys([&](int i, uint32_t key) {
                        if (key >= L) {
                            if (pos < static_cast<unsigned>(kSCCap)) cand[pos] = pack(key, i);
                            ++pos;
                        }
                    });
            }
        } else {
            for_keys([&](int i, uint32_t key) {
                const bool take = key >= L;
                const unsigned act = __activemask();
                const unsigned bal = __ballot_sync(act, take);
                const int leader = __ffs(act) - 1;
                unsigned base = 0;
                if (lane == leader && bal) base = atomicAdd(&sh_count, static_cast<unsigned>(__popc(bal)));
                base = __shfl_sync(act, base, leader);
                if (take) {
                    const unsigned pos = base + __popc(bal & ((1u << lane) - 1u));
                    if (pos < static_cast<unsigned>(kSCCap)) cand[pos] = pack(key, i);
                }
            });
        }
        __syncthreads();
        M = static_cast<int>(sh_count);
        if (M > kSCCap) {
            // too many to hold: the exact kc-th best key T of the chunk (a four-pass radix select),
            // the keys above it, and of the keys equal to T the lowest-index ones
            uint32_t prefix = 0, mask = 0;
            unsigned remain = static_cast<unsigned>(kc);
            for (int pass = 0; pass < 4; ++pass) {
                const int shift = 24 - 8 * pass;
                if (tid < 256) hist[0][tid] = 0u;
                __syncthreads();
                for_keys([&](int, uint32_t key) {
                    if ((key & mask) == prefix) atomicAdd(&hist[0][(key >> shift) & 255u], 1u);
                });
                __syncthreads();
                select_digit(hist[0], prefix, shift, remain);
                __syncthreads();
                prefix = sh_prefix;
                remain = sh_remain;
                mask |= 0xFFu << shift;
            }
            const uint32_t T = prefix;
            const unsigned take_ties = remain;
            const unsigned above_T = static_cast<unsigned>(kc) - take_ties;
            const bool all_ties = sh_ties == take_ties;
            __syncthreads();
            if (tid == 0) { sh_count = 0; sh_tie_base = 0; }
            __syncthreads();
            for_keys([&](int i, uint32_t key) {
                if (key > T) cand[atomicAdd(&sh_count, 1u)] = pack(key, i);
                else if (key == T && all_ties) cand[above_T + atomicAdd(&sh_tie_base, 1u)] = pack(key, i);
            });
            if (!all_ties) {
                // walk the chunk in index order, kSCThreads at a time; a block-wide exclusive scan
                // gives each tie its rank among ties
                __syncthreads();
                unsigned running = 0;
                for (int base = 0; base < len && running < take_ties; base += kSCThreads) {
                    const int i = lo + base + tid;
                    const unsigned flag = (base + tid < len && rank_key(ld_dep_f32(row + i)) == T) ? 1u : 0u;
                    const unsigned bal = __ballot_sync(0xffffffffu, flag);
                    if (lane == 0) warp_sum[warp] = __popc(bal);
                    __syncthreads();
                    unsigned before = 0, total = 0;
                    for (int w = 0; w < kSCThreads / 32; ++w) {
                        const unsigned c = warp_sum[w];
                        if (w < warp) before += c;
                        total += c;
                    }
                    const unsigned r = running + before + __popc(bal & ((1u << lane) - 1u));
                    if (flag && r < take_ties) cand[above_T + r] = pack(T, i);
                    running += total;
                    __syncthreads();
                }
            }
            __syncthreads();
            M = kc;
        }
    }
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // every CTA of the cluster runs
    if (tid >= kc && tid < kClusterMaxK) put(tid, 0ull);          // the padding
    if (kc > 0) {
        if (M <= 256) {
            // rank by counting: the keys are unique, so the ranks are a permutation
            if (tid < M) {
                const unsigned long long x = cand[tid];
                int r = 0;
                for (int j = 0; j < M; ++j) r += cand[j] > x ? 1 : 0;
                if (r < kc) put(r, x);
            }
        } else {
            int P = 1;
            while (P < M) P <<= 1;
            for (int i = M + tid; i < P; i += kSCThreads) cand[i] = 0ull;
            __syncthreads();
            sort_desc(cand, P);
            if (tid < kc) put(tid, cand[tid]);
        }
    }
    cluster_barrier();  // every list is in every CTA's shared memory

    // ---- (2) each CTA ranks its own list's entries among all lists; (3) the entries ranked
    // below k are scored in place, each CTA's best (a shared-memory 64-bit max) goes to the leader,
    // and the best of those picks the token.
    // Thread tid handles entry e = tid / kSC of this CTA's list against list o = tid % kSC: the
    // entries of list o above it, by a branch-free binary search over the list's kClusterMaxK slots
    // (steps 64 .. 1 count among the first 127, the last slot on its own; padding slots hold 0,
    // below every key); the kSC lanes of an entry add their counts with shuffles.
    static_assert(kSC * kClusterMaxK == kSCThreads, "one thread per (entry, list)");
    {
        const int e = tid / kSC, o = tid % kSC;
        const unsigned long long x = my_slots[e];
        const unsigned long long* a = all + o * kListStride;
        int p = 0;
#pragma unroll
        for (int step = kClusterMaxK / 2; step > 0; step >>= 1) p += a[p + step - 1] > x ? step : 0;
        p += a[p] > x ? 1 : 0;
        int rank = o == static_cast<int>(crank) ? e : p;  // its own list: its place in it
#pragma unroll
        for (int d = kSC / 2; d > 0; d >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, d);
        if (o == 0 && e < kc && rank < k) {
            const int idx = static_cast<int>(~static_cast<uint32_t>(x & 0xFFFFFFFFull));
            if (topk) topk[static_cast<size_t>(b) * k + rank] = idx;
            // the logit back from its key (rank_key inverted; -0 comes back as +0 and every NaN as
            // one NaN, which changes no comparison below)
            const uint32_t key = static_cast<uint32_t>(x >> 32);
            const float v = __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
            const float sc = __fadd_rn(__fmul_rn(v, inv_t), s_noise[rank]);
            // the score's key above, the complemented rank below: the largest is the best score,
            // NaN first, the lower rank among equal scores (the q4_sample_kernel rule)
            const unsigned long long sk =
                (static_cast<unsigned long long>(rank_key(sc)) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(rank));
            my_idx[rank] = idx;
            atomicMax(&my_best, sk);
        }
    }
    __syncthreads();
    if (tid == 0) {
        const unsigned long long best = my_best;
        const unsigned long long bidx =
            best ? static_cast<unsigned long long>(my_idx[~static_cast<uint32_t>(best & 0xFFFFFFFFull)]) : 0ull;
        if (crank == 0) {
            cl_best[0] = best;
            cl_idx[0] = bidx;
        } else {
            st_cluster_u64(&cl_best[crank], 0u, best);
            st_cluster_u64(&cl_idx[crank], 0u, bidx);
        }
    }
    cluster_barrier();  // every CTA's best is in the leader's shared memory
    if (crank == 0 && tid == 0) {
        unsigned long long best = cl_best[0], bidx = cl_idx[0];
        for (int c = 1; c < kSC; ++c)
            if (cl_best[c] > best) { best = cl_best[c]; bidx = cl_idx[c]; }
        token[b] = static_cast<int32_t>(bidx);
    }
}

// ================================================================== int4 prefill GEMM
// q4_prefill_kernel: Y[m, n] = sum_k w_hat[n, k] X[m, k] for a prompt of M tokens (the rumik-oss-1
// write-up, "Step 8: a prefill that stays int4": no dequantised copy of the weights; each group is
// expanded in registers for the tensor cores and its scale and minimum are folded into the fp32
// result).  The tokens are
// taken 8 at a time (a "token block"), each block prepared by q4_xprep_kernel exactly like a B = 8
// decode activation (layout LM: scaled per token, group sums divided by the token factor).  A CTA of
// WARPS warps covers WARPS 16-row tiles (one per warp) and TBS token blocks; for every 128-column
// group it stages the TBS blocks' fragments in shared memory (cp.async, double-buffered) while each
// warp loads its tile's record from the tiled copy, unpacks the codes once into 32 operand
// registers and reuses them for 8 mma per token block, then folds scale and minimum in per block:
// acc += scale c + min S'.  y = acc * the token's factor.  Tensor-bound for long prompts: 8 TBS mma
// per 1,088-byte record.

struct PrefillParams {
    const uint8_t* tiled;
    const unsigned char* prep;  // token block b's prepared activations at prep + b * prep_stride
    size_t prep_stride;
    float* y;                   // [M, N]
    int N, K, M;
};

template <int WARPS, int TBS>
__global__ void __launch_bounds__(WARPS * 32) q4_prefill_kernel(const __grid_constant__ PrefillParams p) {
    constexpr int kXs = 4 * 32 * 16;  // one token block's fragments of one group: 2,048 bytes
    __shared__ __align__(16) unsigned char xs[2][TBS][kXs];
    __shared__ __align__(16) float ss[2][TBS][8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = lane & 3, q = lane >> 2;
    const int G = p.K >> 7;
    const int T = (p.N + 15) >> 4;
    const int tile = blockIdx.x * WARPS + warp;
    const bool active = tile < T;
    const int nblk = (p.M + 7) >> 3;
    const int tb0 = blockIdx.y * TBS;
    const int nb = min(TBS, nblk - tb0);  // token blocks of this CTA

    // stage group g's fragments and sums of the CTA's token blocks into buffer `buf`
    auto stage = [&](int g, int buf) {
        constexpr int kChunks = TBS * (kXs / 16 + 2);
        for (int c = threadIdx.x; c < kChunks; c += WARPS * 32) {
            const int b = c / (kXs / 16 + 2), r = c - b * (kXs / 16 + 2);
            if (b >= nb) continue;
            const unsigned char* base = p.prep + (tb0 + b) * p.prep_stride;
            if (r < kXs / 16) {
                cp_async16(&xs[buf][b][16 * r], base + static_cast<size_t>(g) * kXs + 16 * r);
            } else {
                const unsigned char* S = base + static_cast<size_t>(G) * kXs;  // G groups x 8 floats
                cp_async16(&ss[buf][b][4 * (r - kXs / 16)], S + static_cast<size_t>(g) * 32 + 16 * (r - kXs / 16));
            }
        }
        cp_async_commit();
    };

    grid_dependency_wait();  // the prepared activations come from the kernel before
    allow_dependents();

    float acc[TBS][4];
#pragma unroll
    for (int b = 0; b < TBS; ++b) acc[b][0] = acc[b][1] = acc[b][2] = acc[b][3] = 0.f;
    const uint8_t* rec = p.tiled + static_cast<size_t>(active ? tile : 0) * G * kRecBytes;
    // this warp's record of group g (read-only weights) is loaded one group ahead
    uint4 nqa = make_uint4(0u, 0u, 0u, 0u), nqb = nqa;
    uint2 nsc = make_uint2(0u, 0u);
    if (active) {
        nqa = ld_stream_u4(rec + 16 * lane);
        nqb = ld_stream_u4(rec + 512 + 16 * lane);
        nsc = ld_stream_u2(rec + 1024 + 8 * q);
    }
    stage(0, 0);
#pragma unroll 1
    for (int g = 0; g < G; ++g) {
        const int buf = g & 1;
        if (g + 1 < G) stage(g + 1, buf ^ 1);
        else cp_async_commit();  // keep one group per step
        // unpack group g's codes once into 32 operand registers; request group g+1's record
        uint32_t A[8][4];
        const uint4 qa = nqa, qb = nqb;
        const uint2 sc = nsc;
        if (active && g + 1 < G) {
            const uint8_t* r = rec + static_cast<size_t>(g + 1) * kRecBytes;
            nqa = ld_stream_u4(r + 16 * lane);
            nqb = ld_stream_u4(r + 512 + 16 * lane);
            nsc = ld_stream_u2(r + 1024 + 8 * q);
        }
        {
            const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w};
            const uint32_t wb[4] = {qb.x, qb.y, qb.z, qb.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t wa8 = wa[i] >> 8, wb8 = wb[i] >> 8;
                A[2 * i][0] = lo_nibbles(wa[i]);
                A[2 * i][1] = lo_nibbles(wb[i]);
                A[2 * i][2] = hi_nibbles(wa[i]);
                A[2 * i][3] = hi_nibbles(wb[i]);
                A[2 * i + 1][0] = lo_nibbles(wa8);
                A[2 * i + 1][1] = lo_nibbles(wb8);
                A[2 * i + 1][2] = hi_nibbles(wa8);
                A[2 * i + 1][3] = hi_nibbles(wb8);
            }
        }
        cp_async_wait<1>();  // group g's stage has landed
        __syncthreads();
        if (active) {
            const float sa = half_bits_to_f32(sc.x), ma = half_bits_to_f32(sc.x >> 16);
            const float sb = half_bits_to_f32(sc.y), mb = half_bits_to_f32(sc.y >> 16);
#pragma unroll
            for (int b = 0; b < TBS; ++b) {
                if (b < nb) {
                    uint4 xv[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) xv[j] = lds128(&xs[buf][b][(j * 32 + lane) * 16]);
                    float c1[4], c2[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float (&d)[4] = i < 2 ? c1 : c2;
                        if (i == 0 || i == 2)
                            mma_bf16_m16n8k16_zc(d, A[2 * i][0], A[2 * i][1], A[2 * i][2], A[2 * i][3], xv[i].x, xv[i].y);
                        else
                            mma_bf16_m16n8k16(d, A[2 * i][0], A[2 * i][1], A[2 * i][2], A[2 * i][3], xv[i].x, xv[i].y);
                        mma_bf16_m16n8k16(d, A[2 * i + 1][0], A[2 * i + 1][1], A[2 * i + 1][2], A[2 * i + 1][3],
                                          xv[i].z, xv[i].w);
                    }
                    const float2 S = *reinterpret_cast<const float2*>(&ss[buf][b][2 * t]);
                    acc[b][0] = fmaf(sa, c1[0] + c2[0], acc[b][0]);
                    acc[b][0] = fmaf(ma, S.x, acc[b][0]);
                    acc[b][1] = fmaf(sa, c1[1] + c2[1], acc[b][1]);
                    acc[b][1] = fmaf(ma, S.y, acc[b][1]);
                    acc[b][2] = fmaf(sb, c1[2] + c2[2], acc[b][2]);
                    acc[b][2] = fmaf(mb, S.x, acc[b][2]);
                    acc[b][3] = fmaf(sb, c1[3] + c2[3], acc[b][3]);
                    acc[b][3] = fmaf(mb, S.y, acc[b][3]);
                }
            }
        }
        __syncthreads();  // buffer `buf` is restaged in the next step
    }
    cp_async_wait<0>();
    if (!active) return;
    const int ra = 16 * tile + q, rbw = ra + 8;
#pragma unroll
    for (int b = 0; b < TBS; ++b) {
        if (b >= nb) continue;
        const unsigned char* base = p.prep + (tb0 + b) * p.prep_stride;
        const float* fac = reinterpret_cast<const float*>(base + static_cast<size_t>(G) * (kXs + 32));
        const float f0 = ld_dep_f32(fac + 2 * t), f1 = ld_dep_f32(fac + 2 * t + 1);
        const int m0 = 8 * (tb0 + b) + 2 * t, m1 = m0 + 1;
        if (ra < p.N) {
            if (m0 < p.M) p.y[static_cast<size_t>(m0) * p.N + ra] = acc[b][0] * f0;
            if (m1 < p.M) p.y[static_cast<size_t>(m1) * p.N + ra] = acc[b][1] * f1;
        }
        if (rbw < p.N) {
            if (m0 < p.M) p.y[static_cast<size_t>(m0) * p.N + rbw] = acc[b][2] * f0;
            if (m1 < p.M) p.y[static_cast<size_t>(m1) * p.N + rbw] = acc[b][3] * f1;
        }
    }
}

// ================================================================== host
int env_int(const char* name, int dflt) {
    const char* v = std::getenv(name);
    if (!v || !*v) return dflt;
    return std::atoi(v);
}

int device_sm_count(int* dev_out) {
    static int cache[kMaxDevices];
    static std::once_flag flags[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    std::call_once(flags[dev], [dev] {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 0;
        cache[dev] = n;
    });
    if (dev_out) *dev_out = dev;
    return cache[dev] > 0 ? cache[dev] : -1;
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Kernel choice and shape knobs: fixed defaults, overridable for benchmarking only.
// kernel: 0 direct on L1 + tensor cores (default), 1 direct on L0 + tensor cores,
//         2 direct on L0 + CUDA cores, 3 stream on L1 + tensor cores, 4 direct on L1 + CUDA cores.
struct Knobs {
    int kernel;
    int warps, depth;  // direct kernel
    int sw, sd;        // stream kernel: consumer warps, ring stages per consumer warp
    int ksplit_min;
    bool pdl, rotate;
    int l2_ahead;      // direct kernel on L1: units prefetched into L2 ahead of the loads
    int tw, ts;        // tile kernel: warps per CTA and cp.async ring slots per warp
    bool tile_contig;  // tile kernel: record-balanced contiguous shares of the whole list per CTA
};

Knobs knobs() {
    Knobs k{};
    k.kernel = env_int("Q4_KERNEL", -1);  // -1: chosen per call
    if (k.kernel < -1 || k.kernel > 6) k.kernel = -1;
    k.warps = env_int("Q4_WARPS", 16);
    k.depth = env_int("Q4_DEPTH", 4);
    const bool ok = (k.warps == 16 && (k.depth == 2 || k.depth == 4 || k.depth == 6)) ||
                    (k.warps == 8 && (k.depth == 4 || k.depth == 8));
    if (!ok || k.kernel == 2 || k.kernel == 4) { k.warps = 16; k.depth = 4; }
    k.sw = env_int("Q4_SW", 8);
    k.sd = env_int("Q4_SD", 2);
    const bool sok = (k.sw == 8 && (k.sd == 1 || k.sd == 2)) || (k.sw == 4 && k.sd == 4) || (k.sw == 6 && k.sd == 2);
    if (!sok) { k.sw = 8; k.sd = 2; }
    k.ksplit_min = env_int("Q4_KSPLIT", 0);
    k.pdl = env_int("Q4_PDL", 1) != 0;
    k.rotate = env_int("Q4_ROTATE", 1) != 0;
    // measured on the fused 25,088 x 3072 single call at B=1 (8 calls per CUDA graph): 0 14.3 us,
    // 2 13.3, 3 13.3, 4 13.4, 6 13.8, 8 14.1, 16 15.0
    k.l2_ahead = env_int("Q4_L2_AHEAD", 2);
    if (k.l2_ahead < 0 || k.l2_ahead > 64) k.l2_ahead = 2;
    // tile kernel shape: warps per CTA, and ring slots per warp that go with it
    k.tw = env_int("Q4_TW", 32);
    if (k.tw != 16 && k.tw != 24) k.tw = 32;
    k.ts = k.tw == 16 ? 8 : k.tw == 24 ? 6 : 4;
    k.tile_contig = env_int("Q4_TCONTIG", 0) != 0;
    return k;
}

bool uses_l1(int kernel) { return kernel == 0 || kernel == 3 || kernel == 4 || kernel == 5 || kernel == 6; }
bool is_stream(int kernel) { return kernel == 3; }
bool is_tiles(int kernel) { return kernel == 5; }
bool is_flat(int kernel) { return kernel == 6; }

// Workspace of the tile kernel: the prepared activations of one matrix (x fragments, group
// sums, column factors), for batch tile bt.
size_t prep_bytes(int64_t K, int bt) {
    const size_t G = static_cast<size_t>(K / 128);
    return align256(G * 256 * bt + G * 32 + 32);
}

// Flat kernel: warps per CTA, ring slots, CTAs (one per SM, at most one per tile), shared memory
// and workspace.
constexpr int kFlatSlots = 4;
int flat_grid(int64_t N, int sms) {
    const int64_t T = (N + 15) / 16;
    return static_cast<int>(T < sms ? T : sms);
}
// shared memory of a flat launch of fw warps; XS adds the staged activations
size_t flat_smem(int fw, int64_t K, int bt, bool xs) {
    return static_cast<size_t>(fw) * kFlatSlots * kRecBytes + static_cast<size_t>(fw) * 2 * 32 * 16 +
           (xs ? prep_bytes(K, bt) : 0);
}
// Warps per CTA: 32 where the activations of 8 batch columns fit beside the 32 rings, else 16.
// A function of K only (it fixes the split, hence the arithmetic order), never of B.
int flat_warps(int64_t K) { return flat_smem(32, K, 8, true) <= kSmemLimit ? 32 : 16; }
bool flat_xs(int64_t K, int bt) { return flat_smem(flat_warps(K), K, bt, true) <= kSmemLimit; }
// Workspace of a list on the flat kernel: the prepared activations when they do not fit in shared
// memory, a slice per matrix (independent) or one shared slice.
size_t flat_list_bytes(const int64_t* N, const int64_t* K, int n, int bt, bool independent) {
    (void)N;
    size_t sum = 0, one_max = 0;
    for (int i = 0; i < n; ++i) {
        const size_t one = flat_xs(K[i], bt) ? 0 : align256(prep_bytes(K[i], bt));
        sum += one;
        if (one > one_max) one_max = one;
    }
    return independent ? sum : one_max;
}

// The split of one (N, K) matrix.  Depends on N, K, the SM count and the kernel -- never on B.
struct Plan {
    int row_blocks, k_splits;
    int gs_max;             // groups per CTA (largest k-slice)
    int tiles_per_pass;     // stream: tiles whose chunk partials fit in shared memory at once
    int passes;             // stream: passes of the largest row block
    int smax;               // direct: most tiles one warp's range can touch
};

size_t ring_bytes(const Knobs& k) { return static_cast<size_t>(k.sw) * k.sd * kStageBytes + kHdrBytes; }

bool default_shape(const Knobs& k) { return k.warps == 16 && k.depth == 4; }

// Batch tile of the instantiation that runs batch B: the next power of two, or 8 for the
// non-default direct shapes (instantiated for 8 columns only).
int batch_tile(const Knobs& k, int kernel, int B) {
    const int bt = B <= 1 ? 1 : (B <= 2 ? 2 : (B <= 4 ? 4 : 8));
    if (kernel == 5 || kernel == 6) return bt;
    if (is_stream(kernel)) return (k.sw == 8 && k.sd == 2) ? bt : 8;
    return default_shape(k) ? bt : 8;
}

size_t plan_smem(const Knobs& k, int kernel, const Plan& p, int B) {
    const int bt = batch_tile(k, kernel, B);
    const size_t xs = static_cast<size_t>(p.gs_max) * 256 * bt + static_cast<size_t>(p.gs_max) * 32 + 64;
    if (is_stream(kernel)) {
        const int cpt = (p.gs_max + kKC - 1) / kKC;
        return ring_bytes(k) + xs + static_cast<size_t>(p.tiles_per_pass) * cpt * 16 * B * 4;
    }
    return xs + static_cast<size_t>(k.warps) * p.smax * 16 * B * 4;
}

bool make_plan(int64_t N, int64_t K, int sms, const Knobs& k, int kernel, Plan* out) {
    Plan p{};
    const int G = static_cast<int>(K / 128);
    const int64_t T_all = (N + 15) / 16;
    if (is_tiles(kernel) || is_flat(kernel)) {
        p.row_blocks = static_cast<int>(T_all < sms ? T_all : sms);
        p.k_splits = 1;
        p.gs_max = G;
        p.passes = 1;
        *out = p;
        return true;
    }
    int ks = k.ksplit_min > 0 ? k.ksplit_min : 1;
    if (ks > G) ks = G;
    for (;; ++ks) {
        if (ks > G) return false;
        int rb_max = sms / ks;
        if (rb_max < 1) rb_max = 1;
        p.row_blocks = static_cast<int>(T_all < rb_max ? T_all : rb_max);
        p.k_splits = ks;
        const int64_t rows_max =
            uses_l1(kernel) ? 16 * ((T_all + p.row_blocks - 1) / p.row_blocks) : (N + p.row_blocks - 1) / p.row_blocks;
        const int Tm = static_cast<int>((rows_max + 15) / 16);
        p.gs_max = (G + ks - 1) / ks;
        const int gs_min = G / ks;
        p.passes = 1;
        if (is_stream(kernel)) {
            const int cpt = (p.gs_max + kKC - 1) / kKC;
            const size_t fixed = ring_bytes(k) + static_cast<size_t>(p.gs_max) * (256 * kMaxB + 32) + 64;
            const size_t per_tile = static_cast<size_t>(cpt) * 16 * kMaxB * 4;
            if (fixed + per_tile > kSmemLimit) continue;
            size_t tpp = (kSmemLimit - fixed) / per_tile;
            if (tpp > static_cast<size_t>(Tm)) tpp = Tm;
            p.tiles_per_pass = static_cast<int>(tpp);
            p.passes = (Tm + p.tiles_per_pass - 1) / p.tiles_per_pass;
            p.smax = 0;
        } else {
            const int64_t Um = static_cast<int64_t>(Tm) * p.gs_max;
            const int upw = static_cast<int>((Um + k.warps - 1) / k.warps);
            int smax = (upw + gs_min - 1) / gs_min + 1;
            if (smax > Tm) smax = Tm;
            if (smax < 1) smax = 1;
            p.smax = smax;
            p.tiles_per_pass = 0;
            if (plan_smem(k, kernel, p, kMaxB) > kSmemLimit) continue;
        }
        break;
    }
    *out = p;
    return true;
}

size_t plan_ws_bytes(const Plan& p, int64_t N, int B) {
    if (p.k_splits <= 1) return 0;
    return align256(static_cast<size_t>(p.row_blocks) * p.passes * 4) + static_cast<size_t>(p.k_splits) * B * N * 4;
}

size_t job_ws_bytes(const Knobs& k, int kernel, const Plan& p, int64_t N, int64_t K, int B) {
    if (is_tiles(kernel)) return prep_bytes(K, batch_tile(k, kernel, B));
    if (is_flat(kernel)) return flat_list_bytes(&N, &K, 1, batch_tile(k, kernel, B), true);
    return align256(plan_ws_bytes(p, N, B));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool has_l0(const q4_matrix& W) { return W.codes && W.scales && W.mins; }

q4_status check_shape(int64_t N, int64_t K) {
    if (N <= 0) return Q4_ERR_INVALID_ARG;
    if (N > 0x7fffffffLL) return Q4_ERR_UNSUPPORTED_SHAPE;
    if (K <= 0 || K % 128 != 0 || K > kMaxK) return Q4_ERR_UNSUPPORTED_SHAPE;
    return Q4_OK;
}

q4_status check_matrix(const q4_matrix* W) {
    if (!W) return Q4_ERR_INVALID_ARG;
    if (!has_l0(*W) && !W->tiled) return Q4_ERR_INVALID_ARG;
    const q4_status s = check_shape(W->N, W->K);
    if (s != Q4_OK) return s;
    if (has_l0(*W) && (!aligned(W->codes, 16) || !aligned(W->scales, 2) || !aligned(W->mins, 2)))
        return Q4_ERR_MISALIGNED;
    if (W->tiled && !aligned(W->tiled, 16)) return Q4_ERR_MISALIGNED;
    return Q4_OK;
}

q4_status check_io(const uint16_t* X, int B, const float* Y) {
    if (!X || !Y) return Q4_ERR_INVALID_ARG;
    if (B < 1 || B > kMaxB) return Q4_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(Y, 4)) return Q4_ERR_MISALIGNED;
    return Q4_OK;
}

bool fault_injected() { return q4i_fault_injected(); }

template <typename Fn>
bool smem_attr_set(Fn fn, int dev) {
    // cudaFuncSetAttribute once per (kernel, device)
    struct Entry {
        const void* fn;
        int dev;
    };
    static Entry done[512];
    static int n_done = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    const void* key = reinterpret_cast<const void*>(fn);
    for (int i = 0; i < n_done; ++i)
        if (done[i].fn == key && done[i].dev == dev) return true;
    // the raised limit plus the kernel's static shared memory must stay under the per-block maximum
    cudaFuncAttributes fa{};
    int optin = 0;
    bool ok = cudaFuncGetAttributes(&fa, fn) == cudaSuccess &&
              cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
              static_cast<size_t>(optin) > fa.sharedSizeBytes;
    if (ok) {
        size_t lim = static_cast<size_t>(optin) - fa.sharedSizeBytes;
        lim = lim < kSmemLimit ? lim : kSmemLimit;
        ok = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(lim)) ==
             cudaSuccess;
    }
    if (!ok) {
        (void)cudaGetLastError();  // not sticky: clear it so that later checks do not see it
        return false;
    }
    if (n_done < 512) done[n_done++] = Entry{key, dev};
    return true;
}

template <typename Fn, typename... Args>
q4_status launch(Fn fn, int dev, unsigned grid, unsigned block, size_t smem, cudaStream_t stream, bool pdl,
                 Args... args) {
    if (fault_injected()) return Q4_ERR_CUDA;
    // only launches past the default 48 KB need the raised limit (which, with a kernel's static
    // shared memory, must stay under the per-block maximum)
    if (smem > 48 * 1024 && !smem_attr_set(fn, dev)) return Q4_ERR_CUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, args...) == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

using KernelFn = void (*)(Params);

template <int W, int DP, bool TL, bool MM>
KernelFn direct_bt(int bt) {
    switch (bt) {
        case 1: return q4_direct_kernel<W, DP, TL, MM, 1>;
        case 2: return q4_direct_kernel<W, DP, TL, MM, 2>;
        case 4: return q4_direct_kernel<W, DP, TL, MM, 4>;
        default: return q4_direct_kernel<W, DP, TL, MM, 8>;
    }
}

KernelFn pick_kernel(const Knobs& k, int kernel, int B) {
    const int bt = batch_tile(k, kernel, B);
    switch (kernel) {
        case 2: return direct_bt<16, 4, false, false>(bt);
        case 4: return direct_bt<16, 4, true, false>(bt);
        case 3:
            if (k.sw == 8 && k.sd == 1) return q4_stream_kernel<8, 1, true, 8>;
            if (k.sw == 4) return q4_stream_kernel<4, 4, true, 8>;
            if (k.sw == 6) return q4_stream_kernel<6, 2, true, 8>;
            switch (bt) {
                case 1: return q4_stream_kernel<8, 2, true, 1>;
                case 2: return q4_stream_kernel<8, 2, true, 2>;
                case 4: return q4_stream_kernel<8, 2, true, 4>;
                default: return q4_stream_kernel<8, 2, true, 8>;
            }
        case 1:
            if (k.warps == 8) return k.depth == 8 ? q4_direct_kernel<8, 8, false, true, 8> : q4_direct_kernel<8, 4, false, true, 8>;
            if (k.depth == 2) return q4_direct_kernel<16, 2, false, true, 8>;
            if (k.depth == 6) return q4_direct_kernel<16, 6, false, true, 8>;
            return direct_bt<16, 4, false, true>(bt);
        default:
            if (k.warps == 8) return k.depth == 8 ? q4_direct_kernel<8, 8, true, true, 8> : q4_direct_kernel<8, 4, true, true, 8>;
            if (k.depth == 2) return q4_direct_kernel<16, 2, true, true, 8>;
            if (k.depth == 6) return q4_direct_kernel<16, 6, true, true, 8>;
            return direct_bt<16, 4, true, true>(bt);
    }
}

unsigned block_threads(const Knobs& k, int kernel) {
    return static_cast<unsigned>(is_stream(kernel) ? (k.sw + 1) * 32 : k.warps * 32);
}

// The kernel a list runs with: the requested one, moved to the other layout if the matrices
// do not all carry the layout it reads.
// The default: a list of independent matrices runs as one persistent tile-kernel launch (no
// barrier between matrices); a single matrix, or a list whose launches must follow one another,
// runs the direct kernel on the tiled copy, which splits K across the warps of a CTA.
// Independent lists of several matrices: the tile kernel.  One matrix at a time: the flat kernel
// when the matrix has fewer than two 16-row tiles per SM (its split keeps every warp busy), else
// the direct kernel.  A function of the shapes and the SM count only, never of B.
int default_kernel(int n, bool independent, int64_t N = 0, int sms = 0) {
    if (independent && n > 1) return 5;
    return (sms > 0 && (N + 15) / 16 < 2 * static_cast<int64_t>(sms)) ? 6 : 0;
}

q4_status effective_kernel(const Knobs& k, const q4_matrix* mats, int n, bool independent, int sms, int* kernel) {
    bool all_l1 = true, all_l0 = true;
    for (int i = 0; i < n; ++i) {
        all_l1 = all_l1 && mats[i].tiled != nullptr;
        all_l0 = all_l0 && has_l0(mats[i]);
    }
    int kn = k.kernel >= 0 ? k.kernel : default_kernel(n, independent, mats[0].N, sms);
    if (uses_l1(kn) && !all_l1) kn = (kn == 4) ? 2 : 1;
    if (!uses_l1(kn) && !all_l0) kn = (kn == 2) ? 4 : 0;
    if (uses_l1(kn) ? !all_l1 : !all_l0) return Q4_ERR_INVALID_ARG;
    *kernel = kn;
    return Q4_OK;
}

unsigned wait_limit() {
    const int v = env_int("Q4_WAIT_LIMIT", 0);
    return v > 0 ? static_cast<unsigned>(v) : kDefaultWaitLimit;
}

// ---- tile kernel: activation prep and streaming as two launches
// Prepared activations of matrix i live at ws + (sum of prep_bytes of the matrices before it)
// (or at ws for every matrix when `shared` lists run one matrix per launch).
// x8: prepare with the int8 head's pairing (q8_head) instead of the int4 one.
q4_status tiles_prepare(const Knobs& k, const q4_matrix* mats, int n, const uint16_t* const* X, int B, void* ws,
                        bool independent, int dev, cudaStream_t stream, bool x8 = false) {
    const int bt = batch_tile(k, 5, B);
    const int per_launch = independent ? kMaxMats : 1;
    size_t off = 0;
    for (int base = 0; base < n; base += per_launch) {
        const int cnt = n - base < per_launch ? n - base : per_launch;
        PrepParams pp;
        std::memset(&pp, 0, sizeof pp);
        pp.n = cnt;
        pp.B = B;
        for (int i = 0; i < cnt; ++i) {
            const q4_matrix& W = mats[base + i];
            const size_t G = static_cast<size_t>(W.K / 128);
            unsigned char* w = static_cast<unsigned char*>(ws) + (independent ? off : 0);
            if (independent) off += prep_bytes(W.K, bt);
            PrepJob& j = pp.j[i];
            j.x = X[base + i];
            j.K = static_cast<int>(W.K);
            j.xf = reinterpret_cast<uint2*>(w);
            j.S = reinterpret_cast<float*>(w + G * 256 * bt);
            j.fac = j.S + G * 8;
        }
        using PrepFn = void (*)(PrepParams);
        const PrepFn pf = x8 ? (bt == 1 ? q4_xprep_kernel<1, true> : bt == 2 ? q4_xprep_kernel<2, true>
                                : bt == 4 ? q4_xprep_kernel<4, true> : q4_xprep_kernel<8, true>)
                             : (bt == 1 ? q4_xprep_kernel<1> : bt == 2 ? q4_xprep_kernel<2>
                                : bt == 4 ? q4_xprep_kernel<4> : q4_xprep_kernel<8>);
        const q4_status s = launch(pf, dev, static_cast<unsigned>(cnt), static_cast<unsigned>(kPrepThreads), 0, stream, k.pdl, pp);
        if (s != Q4_OK) return s;
    }
    return Q4_OK;
}

q4_status tiles_stream(const Knobs& k, const q4_matrix* mats, int n, float* const* Y, int B, const void* ws,
                       bool independent, int dev, int sms, cudaStream_t stream, bool read_only = false) {
    const int bt = batch_tile(k, 5, B);
    const int per_launch = independent ? kMaxMats : 1;
    size_t off = 0;
    for (int base = 0; base < n; base += per_launch) {
        const int cnt = n - base < per_launch ? n - base : per_launch;
        TileParams tp;
        std::memset(&tp, 0, sizeof tp);
        tp.n_mats = cnt;
        tp.B = B;
        tp.contiguous = k.tile_contig ? 1 : 0;
        int grid = 1;
        for (int i = 0; i < cnt; ++i) {
            const q4_matrix& W = mats[base + i];
            const size_t G = static_cast<size_t>(W.K / 128);
            const unsigned char* w = static_cast<const unsigned char*>(ws) + (independent ? off : 0);
            if (independent) off += prep_bytes(W.K, bt);
            TileMat& m = tp.m[i];
            m.tiled = static_cast<const uint8_t*>(W.tiled);
            m.xf = reinterpret_cast<const uint4*>(w);
            m.S = reinterpret_cast<const float*>(w + G * 256 * bt);
            m.fac = m.S + G * 8;
            m.y = Y[base + i];
            m.N = static_cast<int>(W.N);
            m.K = static_cast<int>(W.K);
            const int64_t T_all = (W.N + 15) / 16;
            m.row_blocks = static_cast<int>(T_all < sms ? T_all : sms);
            m.rot = (k.rotate && independent) ? static_cast<int>((static_cast<int64_t>(base + i) * 37) % m.row_blocks)
                                              : 0;
            if (m.row_blocks > grid) grid = m.row_blocks;
        }
        // The order in which CTAs walk the list (not the arithmetic of any output): longest tiles
        // first, then matrices grouped by shape in the order their shape first appears, so that the
        // last tiles a CTA hands out are short and its warps finish together.
        if (cnt > 1) {
            int first[kMaxMats], idx[kMaxMats];
            for (int i = 0; i < cnt; ++i) {
                idx[i] = i;
                first[i] = i;
                for (int j = 0; j < i; ++j)
                    if (tp.m[j].N == tp.m[i].N && tp.m[j].K == tp.m[i].K) { first[i] = first[j]; break; }
            }
            std::stable_sort(idx, idx + cnt, [&](int a, int b) {
                if (tp.m[a].K != tp.m[b].K) return tp.m[a].K > tp.m[b].K;
                return first[a] < first[b];
            });
            TileMat sorted[kMaxMats];
            for (int i = 0; i < cnt; ++i) sorted[i] = tp.m[idx[i]];
            for (int i = 0; i < cnt; ++i) tp.m[i] = sorted[i];
        }
        if (tp.contiguous) grid = sms;  // every CTA takes a share of the whole list
        using TilesFn = void (*)(TileParams);
        TilesFn tf = nullptr;
        const size_t smem = static_cast<size_t>(k.tw) * k.ts * kRecBytes;
        if (k.tw == 24)
            tf = bt == 1 ? q4_tiles_ring_kernel<24, 6, 1> : bt == 2 ? q4_tiles_ring_kernel<24, 6, 2>
               : bt == 4 ? q4_tiles_ring_kernel<24, 6, 4> : q4_tiles_ring_kernel<24, 6, 8>;
        else if (k.tw == 16)
            tf = bt == 1 ? q4_tiles_ring_kernel<16, 8, 1> : bt == 2 ? q4_tiles_ring_kernel<16, 8, 2>
               : bt == 4 ? q4_tiles_ring_kernel<16, 8, 4> : q4_tiles_ring_kernel<16, 8, 8>;
        else
            tf = bt == 1 ? q4_tiles_ring_kernel<32, 4, 1> : bt == 2 ? q4_tiles_ring_kernel<32, 4, 2>
               : bt == 4 ? q4_tiles_ring_kernel<32, 4, 4> : q4_tiles_ring_kernel<32, 4, 8>;
        if (read_only)  // the twin exists for the default shape only
            tf = bt == 1 ? q4_tiles_ring_kernel<32, 4, 1, true> : bt == 2 ? q4_tiles_ring_kernel<32, 4, 2, true>
               : bt == 4 ? q4_tiles_ring_kernel<32, 4, 4, true> : q4_tiles_ring_kernel<32, 4, 8, true>;
        const unsigned threads = static_cast<unsigned>((read_only ? 32 : k.tw) * 32);
        const size_t smem_l = read_only ? static_cast<size_t>(32) * 4 * kRecBytes : smem;
        const q4_status s = launch(tf, dev, static_cast<unsigned>(grid), threads, smem_l, stream, k.pdl, tp);
        if (s != Q4_OK) return s;
    }
    return Q4_OK;
}

// Each matrix of a list on the flat kernel, one launch per matrix (after an activation prep launch
// when the activations do not fit in shared memory), stream-ordered.  An independent list gives
// every matrix its own workspace slice, a chained one reuses one slice.
q4_status flat_run(const Knobs& k, const q4_matrix* mats, int n, const uint16_t* const* X, float* const* Y, int B,
                   void* ws, bool independent, int dev, int sms, cudaStream_t stream) {
    const int bt = batch_tile(k, 6, B);
    unsigned char* base = static_cast<unsigned char*>(ws);
    for (int i = 0; i < n; ++i) {
        const q4_matrix& W = mats[i];
        const bool xs = flat_xs(W.K, bt);
        const size_t G = static_cast<size_t>(W.K / 128);
        FlatParams fp;
        std::memset(&fp, 0, sizeof fp);
        fp.tiled = static_cast<const uint8_t*>(W.tiled);
        fp.x = X[i];
        fp.y = Y[i];
        fp.N = static_cast<int>(W.N);
        fp.K = static_cast<int>(W.K);
        fp.B = B;
        fp.T = static_cast<int>((W.N + 15) / 16);
        if (!xs) {
            q4_status s = tiles_prepare(k, &W, 1, &X[i], B, base, true, dev, stream);
            if (s != Q4_OK) return s;
            fp.xf = reinterpret_cast<const uint4*>(base);
            fp.S = reinterpret_cast<const float*>(base + G * 256 * bt);
            fp.fac = fp.S + G * 8;
            if (independent) base += align256(prep_bytes(W.K, bt));
        }
        using FlatFn = void (*)(FlatParams);
        const int fw = flat_warps(W.K);
        FlatFn ff;
        if (fw == 32 && xs)
            ff = bt == 1 ? q4_flat_kernel<32, kFlatSlots, 1, true> : bt == 2 ? q4_flat_kernel<32, kFlatSlots, 2, true>
               : bt == 4 ? q4_flat_kernel<32, kFlatSlots, 4, true> : q4_flat_kernel<32, kFlatSlots, 8, true>;
        else if (fw == 32)
            ff = bt == 1 ? q4_flat_kernel<32, kFlatSlots, 1, false> : bt == 2 ? q4_flat_kernel<32, kFlatSlots, 2, false>
               : bt == 4 ? q4_flat_kernel<32, kFlatSlots, 4, false> : q4_flat_kernel<32, kFlatSlots, 8, false>;
        else if (xs)
            ff = bt == 1 ? q4_flat_kernel<16, kFlatSlots, 1, true> : bt == 2 ? q4_flat_kernel<16, kFlatSlots, 2, true>
               : bt == 4 ? q4_flat_kernel<16, kFlatSlots, 4, true> : q4_flat_kernel<16, kFlatSlots, 8, true>;
        else
            ff = bt == 1 ? q4_flat_kernel<16, kFlatSlots, 1, false> : bt == 2 ? q4_flat_kernel<16, kFlatSlots, 2, false>
               : bt == 4 ? q4_flat_kernel<16, kFlatSlots, 4, false> : q4_flat_kernel<16, kFlatSlots, 8, false>;
        const q4_status s = launch(ff, dev, static_cast<unsigned>(flat_grid(W.N, sms)), static_cast<unsigned>(fw * 32),
                                   flat_smem(fw, W.K, bt, xs), stream, k.pdl, fp);
        if (s != Q4_OK) return s;
    }
    return Q4_OK;
}

size_t step_prep_bytes(const int64_t* K, int n, int B) {
    const Knobs k = knobs();
    const int bt = batch_tile(k, 5, B);
    size_t need = 0;
    for (int i = 0; i < n; ++i) need += prep_bytes(K[i], bt);
    return need;
}

// Validate a list, then enqueue it: one persistent launch per kMaxMats matrices when the list
// is independent, else one launch per matrix (stream-ordered, so Y[i] may feed X[j], j > i).
q4_status run(const q4_matrix* mats, int n, const uint16_t* const* X, float* const* Y, int B, void* ws,
              size_t ws_bytes, bool independent, cudaStream_t stream) {
    if (!mats || !X || !Y || n < 1) return Q4_ERR_INVALID_ARG;
    if (B < 1 || B > kMaxB) return Q4_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        q4_status s = check_matrix(&mats[i]);
        if (s != Q4_OK) return s;
        if ((s = check_io(X[i], B, Y[i])) != Q4_OK) return s;
    }
    const Knobs k = knobs();
    int dev = 0;
    const int sms = device_sm_count(&dev);
    if (sms <= 0) return Q4_ERR_CUDA;
    if (!independent && n > 1 && k.kernel < 0) {
        // a chained list runs one matrix per launch anyway: each with its own kernel choice, all in
        // the one workspace slice (stream order keeps them apart)
        for (int i = 0; i < n; ++i) {
            const q4_status s = run(&mats[i], 1, &X[i], &Y[i], B, ws, ws_bytes, true, stream);
            if (s != Q4_OK) return s;
        }
        return Q4_OK;
    }
    int kernel = 0;
    q4_status st = effective_kernel(k, mats, n, independent, sms, &kernel);
    if (st != Q4_OK) return st;
    // plans and workspace: a persistent list gives every k-split matrix its own slice
    size_t need = 0;
    for (int i = 0; i < n; ++i) {
        Plan pl;
        if (!make_plan(mats[i].N, mats[i].K, sms, k, kernel, &pl)) return Q4_ERR_UNSUPPORTED_SHAPE;
        const size_t b = job_ws_bytes(k, kernel, pl, mats[i].N, mats[i].K, B);
        need = independent ? need + b : (b > need ? b : need);
    }
    if (is_flat(kernel)) {
        std::vector<int64_t> Ns(n), Ks(n);
        for (int i = 0; i < n; ++i) { Ns[i] = mats[i].N; Ks[i] = mats[i].K; }
        need = flat_list_bytes(Ns.data(), Ks.data(), n, batch_tile(k, kernel, B), independent);
    }
    if (need > 0) {
        if (!ws || ws_bytes < need) return Q4_ERR_WORKSPACE;
        if (!aligned(ws, 16)) return Q4_ERR_MISALIGNED;
    }
    const int per_launch = independent ? kMaxMats : 1;
    if (is_flat(kernel)) return flat_run(k, mats, n, X, Y, B, ws, independent, dev, sms, stream);
    if (is_tiles(kernel)) {
        q4_status s2 = tiles_prepare(k, mats, n, X, B, ws, independent, dev, stream);
        if (s2 != Q4_OK) return s2;
        return tiles_stream(k, mats, n, Y, B, ws, independent, dev, sms, stream);
    }
    size_t off = 0;
    for (int base = 0; base < n; base += per_launch) {
        const int cnt = n - base < per_launch ? n - base : per_launch;
        Params prm;
        std::memset(&prm, 0, sizeof prm);
        prm.n_mats = cnt;
        prm.B = B;
        prm.wait_limit = wait_limit();
        prm.l2_ahead = k.l2_ahead;
        size_t smem = 0;
        int grid = 1;
        for (int i = 0; i < cnt; ++i) {
            const q4_matrix& W = mats[base + i];
            Plan pl;
            make_plan(W.N, W.K, sms, k, kernel, &pl);
            MatDesc& m = prm.m[i];
            m.codes = W.codes;
            m.scales = W.scales;
            m.mins = W.mins;
            m.tiled = static_cast<const uint8_t*>(W.tiled);
            m.x = X[base + i];
            m.y = Y[base + i];
            m.N = static_cast<int>(W.N);
            m.K = static_cast<int>(W.K);
            m.row_blocks = pl.row_blocks;
            m.k_splits = pl.k_splits;
            m.tiles_per_pass = pl.tiles_per_pass;
            m.passes = pl.passes;
            m.smax = pl.smax;
            m.rot = (k.rotate && independent) ? static_cast<int>((static_cast<int64_t>(base + i) * 37) % pl.row_blocks) : 0;
            if (pl.k_splits > 1) {
                unsigned char* w = static_cast<unsigned char*>(ws) + (independent ? off : 0);
                m.ws_cnt = reinterpret_cast<unsigned*>(w);
                m.ws_part = reinterpret_cast<float*>(w + align256(static_cast<size_t>(pl.row_blocks) * pl.passes * 4));
                if (independent) off += align256(plan_ws_bytes(pl, W.N, B));
            }
            const size_t sm = plan_smem(k, kernel, pl, B);
            if (sm > smem) smem = sm;
            if (pl.row_blocks * pl.k_splits > grid) grid = pl.row_blocks * pl.k_splits;
        }
        if (smem > kSmemLimit) return Q4_ERR_UNSUPPORTED_SHAPE;
        const q4_status s = launch(pick_kernel(k, kernel, B), dev, static_cast<unsigned>(grid),
                                   block_threads(k, kernel), smem, stream, k.pdl, prm);
        if (s != Q4_OK) return s;
    }
    return Q4_OK;
}

// The split (and so the workspace) depends on the kernel family only through the shared-memory
// budget that decides k_splits; the layout (row vs tile grain) does not change it.
size_t workspace_for(const int64_t* N, const int64_t* K, int n, int B, bool independent) {
    if (n < 1 || B < 1 || B > kMaxB) return 0;
    const int sms = device_sm_count(nullptr);
    if (sms <= 0) return 0;
    const Knobs k = knobs();
    if (!independent && n > 1 && k.kernel < 0) {  // one matrix at a time (see run)
        size_t m = 0;
        for (int i = 0; i < n; ++i) {
            const size_t b = workspace_for(&N[i], &K[i], 1, B, true);
            if (check_shape(N[i], K[i]) != Q4_OK) return 0;
            m = b > m ? b : m;
        }
        return m;
    }
    const int kernel = k.kernel >= 0 ? k.kernel : default_kernel(n, independent, N[0], sms);
    // the flat kernel falls back to kernel 1 for matrices without a tiled copy: cover both
    const int kernel2 = is_flat(kernel) ? 1 : kernel;
    size_t need = 0;
    for (int i = 0; i < n; ++i) {
        if (check_shape(N[i], K[i]) != Q4_OK) return 0;
        Plan p;
        if (!make_plan(N[i], K[i], sms, k, kernel2, &p)) return 0;
        const size_t b = job_ws_bytes(k, kernel2, p, N[i], K[i], B);
        need = independent ? need + b : (b > need ? b : need);
    }
    if (is_flat(kernel)) {
        const size_t f = flat_list_bytes(N, K, n, batch_tile(k, kernel, B), independent);
        if (f > need) need = f;
    }
    return need;
}

}  // namespace

int q4i_sm_count(int* dev_out) { return device_sm_count(dev_out); }

bool q4i_fault_injected() {
    const char* v = std::getenv("Q4_FAULT_INJECT");
    return v && std::strcmp(v, "launch") == 0;
}

// ------------------------------------------------------------------ C ABI
extern "C" size_t q4_tiled_bytes(int64_t N, int64_t K) {
    if (check_shape(N, K) != Q4_OK) return 0;
    return static_cast<size_t>((N + 15) / 16) * static_cast<size_t>(K / 128) * kRecBytes;
}

extern "C" q4_status q4_tile(const q4_matrix* W, void* tiled, size_t tiled_bytes, void* stream) {
    if (!W || !has_l0(*W) || !tiled) return Q4_ERR_INVALID_ARG;
    q4_status s = check_shape(W->N, W->K);
    if (s != Q4_OK) return s;
    if (!aligned(W->codes, 16) || !aligned(W->scales, 2) || !aligned(W->mins, 2) || !aligned(tiled, 16))
        return Q4_ERR_MISALIGNED;
    if (tiled_bytes < q4_tiled_bytes(W->N, W->K)) return Q4_ERR_WORKSPACE;
    if (fault_injected()) return Q4_ERR_CUDA;
    const int64_t pieces = ((W->N + 15) / 16) * (W->K / 128) * 68;
    const unsigned grid = static_cast<unsigned>((pieces + 255) / 256);
    q4_tile_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        W->codes, W->scales, W->mins, static_cast<int>(W->N), static_cast<int>(W->K), static_cast<uint8_t*>(tiled),
        pieces);
    return cudaPeekAtLastError() == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

extern "C" size_t q4_workspace_bytes(int64_t N, int64_t K, int B) {
    return workspace_for(&N, &K, 1, B, true);
}

extern "C" size_t q4_decode_step_workspace_bytes(const int64_t* N, const int64_t* K, int n_mats, int B,
                                                 unsigned flags) {
    if (!N || !K) return 0;
    return workspace_for(N, K, n_mats, B, (flags & Q4_STEP_INDEPENDENT) != 0);
}

extern "C" q4_status q4_plan(int64_t N, int64_t K, q4_plan_info* out) {
    if (!out) return Q4_ERR_INVALID_ARG;
    const q4_status s = check_shape(N, K);
    if (s != Q4_OK) return s;
    const int sms = device_sm_count(nullptr);
    if (sms <= 0) return Q4_ERR_CUDA;
    Knobs k = knobs();
    if (k.kernel < 0) k.kernel = default_kernel(1, true, N, sms);
    Plan p;
    if (!make_plan(N, K, sms, k, k.kernel, &p)) return Q4_ERR_UNSUPPORTED_SHAPE;
    out->row_blocks = p.row_blocks;
    out->k_splits = p.k_splits;
    out->warps_per_cta = is_tiles(k.kernel)  ? k.tw
                         : is_flat(k.kernel) ? flat_warps(K)
                                             : static_cast<int32_t>(block_threads(k, k.kernel) / 32);
    out->prefetch_depth = is_stream(k.kernel) ? k.sw * k.sd : k.depth;
    out->kernel = k.kernel;
    out->sm_count = sms;
    return Q4_OK;
}

extern "C" q4_status q4_gemm_skinny(const q4_matrix* W, const uint16_t* X, int B, float* Y, void* ws,
                                    size_t ws_bytes, void* stream) {
    if (!W) return Q4_ERR_INVALID_ARG;
    q4_status s = check_matrix(W);
    if (s != Q4_OK) return s;
    if ((s = check_io(X, B, Y)) != Q4_OK) return s;
    return run(W, 1, &X, &Y, B, ws, ws_bytes, true, static_cast<cudaStream_t>(stream));
}

extern "C" q4_status q4_gemv(const q4_matrix* W, const uint16_t* x, float* y, void* ws, size_t ws_bytes,
                             void* stream) {
    return q4_gemm_skinny(W, x, 1, y, ws, ws_bytes, stream);
}

extern "C" q4_status q4_decode_step(const q4_matrix* mats, int n_mats, const uint16_t* const* X,
                                    float* const* Y, int B, void* ws, size_t ws_bytes, unsigned flags,
                                    void* stream) {
    return run(mats, n_mats, X, Y, B, ws, ws_bytes, (flags & Q4_STEP_INDEPENDENT) != 0,
               static_cast<cudaStream_t>(stream));
}

extern "C" size_t q4_step_workspace_bytes(const int64_t* K, int n_mats, int B) {
    if (!K || n_mats < 1 || B < 1 || B > kMaxB) return 0;
    for (int i = 0; i < n_mats; ++i)
        if (K[i] <= 0 || K[i] % 128 || K[i] > kMaxK) return 0;
    return step_prep_bytes(K, n_mats, B);
}

// Shared checks of the two phases.
static q4_status check_step(const q4_matrix* mats, int n, int B, const void* ws, size_t ws_bytes, int* dev, int* sms) {
    if (!mats || n < 1 || B < 1 || B > kMaxB || !ws) return Q4_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        const q4_status s = check_matrix(&mats[i]);
        if (s != Q4_OK) return s;
        if (!mats[i].tiled) return Q4_ERR_INVALID_ARG;
    }
    if (!aligned(ws, 16)) return Q4_ERR_MISALIGNED;
    size_t need = 0;
    const Knobs k = knobs();
    for (int i = 0; i < n; ++i) need += prep_bytes(mats[i].K, batch_tile(k, 5, B));
    if (ws_bytes < need) return Q4_ERR_WORKSPACE;
    *sms = device_sm_count(dev);
    return *sms > 0 ? Q4_OK : Q4_ERR_CUDA;
}

extern "C" q4_status q4_step_prepare(const q4_matrix* mats, int n_mats, const uint16_t* const* X, int B, void* ws,
                                     size_t ws_bytes, void* stream) {
    int dev = 0, sms = 0;
    q4_status s = check_step(mats, n_mats, B, ws, ws_bytes, &dev, &sms);
    if (s != Q4_OK) return s;
    if (!X) return Q4_ERR_INVALID_ARG;
    for (int i = 0; i < n_mats; ++i) {
        if (!X[i]) return Q4_ERR_INVALID_ARG;
        if (!aligned(X[i], 16)) return Q4_ERR_MISALIGNED;
    }
    return tiles_prepare(knobs(), mats, n_mats, X, B, ws, true, dev, static_cast<cudaStream_t>(stream));
}

extern "C" q4_status q4_step_stream(const q4_matrix* mats, int n_mats, float* const* Y, int B, const void* ws,
                                    size_t ws_bytes, void* stream) {
    int dev = 0, sms = 0;
    q4_status s = check_step(mats, n_mats, B, ws, ws_bytes, &dev, &sms);
    if (s != Q4_OK) return s;
    if (!Y) return Q4_ERR_INVALID_ARG;
    for (int i = 0; i < n_mats; ++i) {
        if (!Y[i]) return Q4_ERR_INVALID_ARG;
        if (!aligned(Y[i], 4)) return Q4_ERR_MISALIGNED;
    }
    return tiles_stream(knobs(), mats, n_mats, Y, B, ws, true, dev, sms, static_cast<cudaStream_t>(stream));
}

extern "C" q4_status q4_step_stream_readonly(const q4_matrix* mats, int n_mats, float* const* Y, int B,
                                             const void* ws, size_t ws_bytes, void* stream) {
    int dev = 0, sms = 0;
    const q4_status s = check_step(mats, n_mats, B, ws, ws_bytes, &dev, &sms);
    if (s != Q4_OK) return s;
    if (!Y) return Q4_ERR_INVALID_ARG;
    for (int i = 0; i < n_mats; ++i) {
        if (!Y[i]) return Q4_ERR_INVALID_ARG;
        if (!aligned(Y[i], 4)) return Q4_ERR_MISALIGNED;
    }
    return tiles_stream(knobs(), mats, n_mats, Y, B, ws, true, dev, sms, static_cast<cudaStream_t>(stream), true);
}

// ------------------------------------------------------------------ no-allocation variant
// Scratch of q4_gemm_skinny_noalloc: the prepared activations of one matrix, in device memory
// that the library owns.  Every GPU that loads the library holds these 512 KiB until the process
// exits.  Host code must not pass the symbol itself to a kernel (on the host it names a host-side
// stand-in); the device address is looked up per device with cudaGetSymbolAddress.
static constexpr size_t kNoallocScratchBytes = 512 * 1024;
static __device__ __align__(256) unsigned char g_q4_noalloc_scratch[kNoallocScratchBytes];

// Device address of the scratch on the current device, looked up (with that device current) on
// the first call that finds none cached; nullptr if the lookup failed.  Only a successful lookup is
// kept, so a failed one (say, one made during stream capture) is tried again by the next call.  A
// device reset invalidates the cached address: the process must not reset a device it uses this on.
static void* noalloc_scratch(int dev) {
    static void* addr[kMaxDevices];
    static std::mutex mu;
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_q4_noalloc_scratch) == cudaSuccess) {
            addr[dev] = p;
        } else {
            (void)cudaGetLastError();  // not sticky: clear it so that later checks do not see it
        }
    }
    return addr[dev];
}

extern "C" size_t q4_noalloc_scratch_bytes(void) { return kNoallocScratchBytes; }

extern "C" q4_status q4_gemm_skinny_noalloc(const q4_matrix* W, const uint16_t* X, int B, float* Y,
                                            void* stream) {
    if (!W) return Q4_ERR_INVALID_ARG;
    q4_status s = check_matrix(W);
    if (s != Q4_OK) return s;
    if (!W->tiled) return Q4_ERR_INVALID_ARG;
    if ((s = check_io(X, B, Y)) != Q4_OK) return s;
    const Knobs k = knobs();
    if (prep_bytes(W->K, batch_tile(k, 5, B)) > kNoallocScratchBytes) return Q4_ERR_WORKSPACE;
    if (fault_injected()) return Q4_ERR_CUDA;
    int dev = 0;
    const int sms = device_sm_count(&dev);
    if (sms <= 0) return Q4_ERR_CUDA;
    void* scratch = noalloc_scratch(dev);
    if (!scratch) return Q4_ERR_CUDA;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    s = tiles_prepare(k, W, 1, &X, B, scratch, true, dev, st);
    if (s != Q4_OK) return s;
    return tiles_stream(k, W, 1, &Y, B, scratch, true, dev, sms, st);
}

// ------------------------------------------------------------------ int4 prefill GEMM
namespace {
size_t prefill_ws(int64_t K, int64_t M) {
    return static_cast<size_t>((M + 7) / 8) * prep_bytes(K, 8);
}
}  // namespace

extern "C" size_t q4_prefill_workspace_bytes(int64_t K, int64_t M) {
    if (K <= 0 || K % 128 != 0 || M < 1 || M > (1 << 24)) return 0;
    const size_t a = prefill_ws(K, M), b = q4i_prefill_tc_ws(K, M);  // enough for either kernel
    return a > b ? a : b;
}

extern "C" int q4_prefill_kernel(int64_t K, int64_t M) {
    if (K <= 0 || K % 128 != 0 || K > kMaxK || M < 1 || M > (1 << 24)) return -1;
    return q4i_prefill_tc_usable(K, M) ? 1 : 0;
}

extern "C" q4_status q4_gemm_prefill(const q4_matrix* W, const uint16_t* X, int64_t M, float* Y, void* ws,
                                     size_t ws_bytes, void* stream) {
    if (!W || !W->tiled || !X || !Y || M < 1 || M > (1 << 24)) return Q4_ERR_INVALID_ARG;
    q4_status st = check_shape(W->N, W->K);
    if (st != Q4_OK) return st;
    if (!aligned(W->tiled, 16) || !aligned(X, 16) || !aligned(Y, 4)) return Q4_ERR_MISALIGNED;
    const bool tc = q4i_prefill_tc_usable(W->K, M);
    const size_t need = tc ? q4i_prefill_tc_ws(W->K, M) : prefill_ws(W->K, M);
    if (!ws || ws_bytes < need) return Q4_ERR_WORKSPACE;
    if (!aligned(ws, 16)) return Q4_ERR_MISALIGNED;
    if (fault_injected()) return Q4_ERR_CUDA;
    int dev = 0;
    if (device_sm_count(&dev) <= 0) return Q4_ERR_CUDA;
    const Knobs k = knobs();
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // on a tcgen05 device: the tensor-memory kernel (q4_prefill_tc.cu)
    if (tc) return q4i_prefill_tc(W, X, M, Y, ws, ws_bytes, cs, k.pdl);
    const size_t stride = prep_bytes(W->K, 8);
    const size_t G = static_cast<size_t>(W->K / 128);
    const int64_t nblk = (M + 7) / 8;
    unsigned char* base = static_cast<unsigned char*>(ws);
    // activations: one prep job per token block of 8 (the last one may hold fewer tokens)
    for (int64_t b0 = 0; b0 < nblk;) {
        const int64_t full_end = M / 8;  // blocks [0, full_end) hold 8 tokens
        const bool partial = b0 >= full_end;
        int64_t b1 = partial ? b0 + 1 : (b0 + kMaxMats < full_end ? b0 + kMaxMats : full_end);
        PrepParams pp;
        std::memset(&pp, 0, sizeof pp);
        pp.n = static_cast<int>(b1 - b0);
        pp.B = partial ? static_cast<int>(M - 8 * b0) : 8;
        for (int64_t b = b0; b < b1; ++b) {
            PrepJob& j = pp.j[b - b0];
            unsigned char* w = base + static_cast<size_t>(b) * stride;
            j.x = X + static_cast<size_t>(b) * 8 * W->K;
            j.K = static_cast<int>(W->K);
            j.xf = reinterpret_cast<uint2*>(w);
            j.S = reinterpret_cast<float*>(w + G * 256 * 8);
            j.fac = j.S + G * 8;
        }
        st = launch(q4_xprep_kernel<8>, dev, static_cast<unsigned>(pp.n), static_cast<unsigned>(kPrepThreads), 0, cs, k.pdl, pp);
        if (st != Q4_OK) return st;
        b0 = b1;
    }
    PrefillParams fp;
    std::memset(&fp, 0, sizeof fp);
    fp.tiled = static_cast<const uint8_t*>(W->tiled);
    fp.prep = base;
    fp.prep_stride = stride;
    fp.y = Y;
    fp.N = static_cast<int>(W->N);
    fp.K = static_cast<int>(W->K);
    fp.M = static_cast<int>(M);
    // CTA tile: 8 row tiles x 8 token blocks; 4 x 4 when that would leave SMs without a CTA (small
    // matrices with short prompts)
    const int64_t T = (W->N + 15) / 16;
    const int sms = device_sm_count(nullptr);
    const bool small = ((T + 7) / 8) * ((nblk + 7) / 8) < sms;
    const int pw = small ? 4 : 8, ptb = small ? 4 : 8;
    const dim3 grid(static_cast<unsigned>((T + pw - 1) / pw), static_cast<unsigned>((nblk + ptb - 1) / ptb));
    if (grid.y > 65535) return Q4_ERR_UNSUPPORTED_SHAPE;
    using PfFn = void (*)(PrefillParams);
    const PfFn pf = small ? q4_prefill_kernel<4, 4> : q4_prefill_kernel<8, 8>;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(pw * 32);
    cfg.stream = cs;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = k.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, pf, fp) == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

// ------------------------------------------------------------------ the int8 head
namespace {
// warps per CTA (16 with 4 ring slots, or 24 with 3) and L2 prefetch distance of the int8 head
int q8_warps() { return env_int("Q4_Q8W", 16) == 24 ? 24 : 16; }
int q8_slots(int w) { return w == 24 ? 3 : 4; }
int q8_pf() {
    const int v = env_int("Q4_Q8PF", 0);
    return v < 0 || v > 64 ? 0 : v;
}
size_t q8_smem(int64_t K, int bt, bool xs) {
    const int w = q8_warps();
    return static_cast<size_t>(w) * q8_slots(w) * kRec8Bytes + static_cast<size_t>(w) * 2 * 32 * 16 +
           (xs ? prep_bytes(K, bt) : 0);
}
bool q8_xs(int64_t K, int bt) { return q8_smem(K, bt, true) <= kSmemLimit; }
size_t q8_cand_bytes(int grid) { return align256(static_cast<size_t>(grid) * 8 * sizeof(int2)); }
size_t q8_ws(int64_t N, int64_t K, int bt, int sms) {
    return q8_cand_bytes(flat_grid(N, sms)) + (q8_xs(K, bt) ? 0 : align256(prep_bytes(K, bt)));
}
int q8_bt(int B) { return B <= 1 ? 1 : (B <= 2 ? 2 : (B <= 4 ? 4 : 8)); }
}  // namespace

extern "C" size_t q8_tiled_bytes(int64_t N, int64_t K) {
    if (check_shape(N, K) != Q4_OK) return 0;
    return static_cast<size_t>((N + 15) / 16) * static_cast<size_t>(K / 128) * kRec8Bytes;
}

extern "C" q4_status q8_tile(const q8_matrix* W, void* tiled, size_t tiled_bytes, void* stream) {
    if (!W || !W->codes || !tiled) return Q4_ERR_INVALID_ARG;
    q4_status s = check_shape(W->N, W->K);
    if (s != Q4_OK) return s;
    if (!aligned(W->codes, 16) || !aligned(tiled, 16)) return Q4_ERR_MISALIGNED;
    if (tiled_bytes < q8_tiled_bytes(W->N, W->K)) return Q4_ERR_WORKSPACE;
    if (fault_injected()) return Q4_ERR_CUDA;
    const int64_t pieces = ((W->N + 15) / 16) * (W->K / 128) * 128;
    const unsigned grid = static_cast<unsigned>((pieces + 255) / 256);
    q8_tile_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        W->codes, static_cast<int>(W->N), static_cast<int>(W->K), static_cast<uint8_t*>(tiled), pieces);
    return cudaPeekAtLastError() == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

extern "C" size_t q8_head_workspace_bytes(int64_t N, int64_t K, int B) {
    if (check_shape(N, K) != Q4_OK || B < 1 || B > kMaxB) return 0;
    const int sms = device_sm_count(nullptr);
    if (sms <= 0) return 0;
    return q8_ws(N, K, q8_bt(B), sms);
}

extern "C" q4_status q8_head(const q8_matrix* W, const uint16_t* X, int B, float* Y, int32_t* idx, void* ws,
                             size_t ws_bytes, void* stream) {
    if (!W || !W->tiled || !W->scales || !X || (!Y && !idx)) return Q4_ERR_INVALID_ARG;
    if (B < 1 || B > kMaxB) return Q4_ERR_INVALID_ARG;
    q4_status st = check_shape(W->N, W->K);
    if (st != Q4_OK) return st;
    if (!aligned(W->tiled, 16) || !aligned(W->scales, 2) || !aligned(X, 16) || (Y && !aligned(Y, 4)) ||
        (idx && !aligned(idx, 4)))
        return Q4_ERR_MISALIGNED;
    int dev = 0;
    const int sms = device_sm_count(&dev);
    if (sms <= 0) return Q4_ERR_CUDA;
    const int bt = q8_bt(B);
    const size_t need = q8_ws(W->N, W->K, bt, sms);
    if (!ws || ws_bytes < need) return Q4_ERR_WORKSPACE;
    if (!aligned(ws, 16)) return Q4_ERR_MISALIGNED;
    if (fault_injected()) return Q4_ERR_CUDA;
    const Knobs k = knobs();
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int grid = flat_grid(W->N, sms);
    const bool xs = q8_xs(W->K, bt);
    unsigned char* w = static_cast<unsigned char*>(ws);
    FlatParams fp;
    std::memset(&fp, 0, sizeof fp);
    fp.tiled = static_cast<const uint8_t*>(W->tiled);
    fp.x = X;
    fp.y = Y;
    fp.rscale = W->scales;
    fp.cand = idx ? reinterpret_cast<int2*>(w) : nullptr;
    fp.N = static_cast<int>(W->N);
    fp.K = static_cast<int>(W->K);
    fp.B = B;
    fp.T = static_cast<int>((W->N + 15) / 16);
    if (!xs) {
        unsigned char* pw = w + q8_cand_bytes(grid);
        q4_matrix m{};
        m.N = W->N;
        m.K = W->K;
        st = tiles_prepare(k, &m, 1, &X, B, pw, true, dev, cs, true);
        if (st != Q4_OK) return st;
        const size_t G = static_cast<size_t>(W->K / 128);
        fp.xf = reinterpret_cast<const uint4*>(pw);
        fp.S = reinterpret_cast<const float*>(pw + G * 256 * bt);
        fp.fac = fp.S + G * 8;
    }
    fp.pf = q8_pf();
    const int qw = q8_warps();
    using FlatFn = void (*)(FlatParams);
    FlatFn ff;
    if (qw == 24 && xs)
        ff = bt == 1 ? q4_flat_kernel<24, 3, 1, true, true> : bt == 2 ? q4_flat_kernel<24, 3, 2, true, true>
           : bt == 4 ? q4_flat_kernel<24, 3, 4, true, true> : q4_flat_kernel<24, 3, 8, true, true>;
    else if (qw == 24)
        ff = bt == 1 ? q4_flat_kernel<24, 3, 1, false, true> : bt == 2 ? q4_flat_kernel<24, 3, 2, false, true>
           : bt == 4 ? q4_flat_kernel<24, 3, 4, false, true> : q4_flat_kernel<24, 3, 8, false, true>;
    else if (xs)
        ff = bt == 1 ? q4_flat_kernel<16, 4, 1, true, true> : bt == 2 ? q4_flat_kernel<16, 4, 2, true, true>
           : bt == 4 ? q4_flat_kernel<16, 4, 4, true, true> : q4_flat_kernel<16, 4, 8, true, true>;
    else
        ff = bt == 1 ? q4_flat_kernel<16, 4, 1, false, true> : bt == 2 ? q4_flat_kernel<16, 4, 2, false, true>
           : bt == 4 ? q4_flat_kernel<16, 4, 4, false, true> : q4_flat_kernel<16, 4, 8, false, true>;
    st = launch(ff, dev, static_cast<unsigned>(grid), static_cast<unsigned>(qw * 32), q8_smem(W->K, bt, xs), cs,
                k.pdl, fp);
    if (st != Q4_OK || !idx) return st;
    return launch(q8_argmax_final, dev, 1u, 256u, 0, cs, k.pdl, static_cast<const int2*>(fp.cand), grid, B, idx);
}

extern "C" q4_status q4_sample_topk(const float* Y, int B, int64_t N, int k, float inv_temperature,
                                    const float* noise, int32_t* token, int32_t* topk, void* stream) {
    if (!Y || !noise || !token || B < 1 || B > 65535 || N < 1 || N > 0x7fffffffLL) return Q4_ERR_INVALID_ARG;
    if (k < 1 || k > kSampleMaxK || k > N) return Q4_ERR_INVALID_ARG;
    if (!(inv_temperature > 0.f) || !std::isfinite(inv_temperature)) return Q4_ERR_INVALID_ARG;
    if (!aligned(Y, 4) || !aligned(noise, 4) || !aligned(token, 4) || (topk && !aligned(topk, 4)))
        return Q4_ERR_MISALIGNED;
    if (fault_injected()) return Q4_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return Q4_ERR_CUDA;
    const bool vec = aligned(Y, 16) && (N % 4) == 0;
    const Knobs kn = knobs();
    if (k <= kClusterMaxK && env_int("Q4_SAMPLE_CLUSTER", 1) != 0) {
        // one cluster of kSC CTAs per row
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(kSC, static_cast<unsigned>(B));
        cfg.blockDim = dim3(kSCThreads);
        cfg.stream = static_cast<cudaStream_t>(stream);
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = kn.pdl ? 1 : 0;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = kSC;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        const bool reg = (((N + kSC - 1) / kSC + 3) & ~int64_t{3}) <= int64_t{kSCThreads} * kSCRegs;
        auto cf = vec ? (reg ? q4_sample_cluster_kernel<true, true> : q4_sample_cluster_kernel<true, false>)
                      : (reg ? q4_sample_cluster_kernel<false, true> : q4_sample_cluster_kernel<false, false>);
        return cudaLaunchKernelEx(&cfg, cf, Y, static_cast<int>(N), k, inv_temperature, noise, token, topk) ==
                       cudaSuccess
                   ? Q4_OK
                   : Q4_ERR_CUDA;
    }
    auto fn = vec ? q4_sample_kernel<true> : q4_sample_kernel<false>;
    return launch(fn, dev, static_cast<unsigned>(B), static_cast<unsigned>(kSampleThreads), 0,
                  static_cast<cudaStream_t>(stream), kn.pdl, Y, static_cast<int>(N), k, inv_temperature, noise, token,
                  topk);
}

extern "C" q4_status q4_argmax_f32(const float* Y, int B, int64_t N, int32_t* idx, void* stream) {
    if (!Y || !idx || B < 1 || B > kMaxB || N < 1 || N > 0x7fffffffLL) return Q4_ERR_INVALID_ARG;
    if (!aligned(Y, 4) || !aligned(idx, 4)) return Q4_ERR_MISALIGNED;
    if (fault_injected()) return Q4_ERR_CUDA;
    const bool cl = env_int("Q4_ARGMAX_CLUSTER", 1) != 0;  // 0: one CTA per row (q4_argmax_kernel)
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = cl ? dim3(kAC, static_cast<unsigned>(B)) : dim3(static_cast<unsigned>(B));
    cfg.blockDim = dim3(cl ? kACThreads : 1024);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = env_int("Q4_PDL", 1) != 0 ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = kAC;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, cl ? q4_argmax_cluster_kernel : q4_argmax_kernel, Y, static_cast<int>(N), idx) ==
                   cudaSuccess
               ? Q4_OK
               : Q4_ERR_CUDA;
}

extern "C" q4_status q4_argmax_key_f32(const float* Y, int B, int64_t N, int64_t index_base, int64_t* keys,
                                       void* stream) {
    if (!Y || !keys || B < 1 || B > 65535 || N < 1 || N > 0x7fffffffLL) return Q4_ERR_INVALID_ARG;
    if (index_base < 0 || index_base + N > 0xFFFFFFFFLL) return Q4_ERR_INVALID_ARG;
    if (!aligned(Y, 4) || !aligned(keys, 8)) return Q4_ERR_MISALIGNED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return Q4_ERR_CUDA;
    return launch(q4_argmax_key_kernel, dev, static_cast<unsigned>(B), 1024u, 0, static_cast<cudaStream_t>(stream),
                  env_int("Q4_PDL", 1) != 0, Y, static_cast<int>(N), static_cast<uint32_t>(index_base), keys);
}

extern "C" q4_status q4_argmax_key_index(const int64_t* keys, int B, int32_t* idx, void* stream) {
    if (!keys || !idx || B < 1 || B > 65535) return Q4_ERR_INVALID_ARG;
    if (!aligned(keys, 8) || !aligned(idx, 4)) return Q4_ERR_MISALIGNED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return Q4_ERR_CUDA;
    return launch(q4_argmax_key_index_kernel, dev, static_cast<unsigned>((B + 255) / 256), 256u, 0,
                  static_cast<cudaStream_t>(stream), env_int("Q4_PDL", 1) != 0, keys, B, idx);
}

extern "C" q4_status q4_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return Q4_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_q4_device_error, sizeof v) != cudaSuccess) return Q4_ERR_CUDA;
    const int attn = q4i_attn_take_error();
    if (attn < 0) return Q4_ERR_CUDA;
    const int pre = q4i_prefill_take_error();
    if (pre < 0) return Q4_ERR_CUDA;
    if (v == 0 && attn == 0 && pre == 0) return Q4_OK;
    if (v == 0) return Q4_ERR_TIMEOUT;
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_q4_device_error, &zero, sizeof zero) != cudaSuccess) return Q4_ERR_CUDA;
    return Q4_ERR_TIMEOUT;
}
