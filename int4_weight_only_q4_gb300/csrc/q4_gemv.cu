// int4 group-128 weight-only GEMV / skinny GEMM (batch 1..8) for GB300, sm_103a.
//
// What is computed (rumik-oss-1 int4 engine page, rtts.neoandmatrix.me,
// "Step 3" and "Step 7"): Y[b, n] = sum_k (code[n,k] * scale[n,g] + min[n,g]) * X[b,k],
// g = k / 128, fp32 accumulation.  Every group is evaluated in the folded form
//     scale * (sum_k (128 + code) x_k)  +  (min - 128 * scale) * (sum_k x_k)
// so that a code becomes a bf16 operand with one LOP3 (128 + code has the bf16
// bit pattern 0x4300 | code; the same exponent-field trick the page's CUDA
// kernel uses with fp16, here with bf16 so it pairs with bf16 activations).
//
// Work split (depends on N, K and the SM count only -- never on B):
//   grid = row_blocks x k_splits CTAs, one per SM.  CTA (rb, ks) owns rows
//   [N*rb/RB, N*(rb+1)/RB) and groups [G*ks/KS, G*(ks+1)/KS).  Its rows form
//   16-row tiles; the (tile, group) units are dealt to the warps in equal
//   contiguous ranges; a warp's partial sums per tile go to shared memory and
//   are added in warp order.  With k_splits > 1 the CTA partials go to the
//   workspace and the last CTA of the row block (arrival ticket) adds them in
//   k-split order.  Every addition order is therefore fixed by (N, K, SMs),
//   which makes each batch column bit-identical to the batch-1 result (the
//   pure-C TTS engine page, wpnews.pro: match the accumulation order).
//
// Per unit a lane streams 16 bytes of codes of row q and of row q+8 of its
// tile (q = lane/4) with 128-bit non-allocating loads, DEPTH units ahead.
// Activations are staged once per CTA in shared memory in the order of the
// mma B fragment, with the per-group sums of x.
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "q4.h"

namespace {

constexpr int kMaxB = 8;
constexpr int64_t kMaxK = 65536;
constexpr int kMaxDevices = 64;
constexpr size_t kSmemLimit = 220 * 1024;  // dynamic; leaves room for static smem under the 227 KB cap

struct GemvArgs {
    const uint8_t* codes;
    const uint16_t* scales;
    const uint16_t* mins;
    const uint16_t* x;
    float* y;
    float* ws_part;          // [k_splits][B][N] when k_splits > 1
    unsigned int* ws_cnt;    // [row_blocks]
    int N, K, B;
    int row_blocks, k_splits, smax;
    int l2_prefetch;         // bytes of this CTA's codes to bulk-prefetch into L2 up front
};

// ------------------------------------------------------------------ device helpers
__device__ __forceinline__ uint4 ld_stream_u4(const uint8_t* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_nc_u16(const uint16_t* p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// bf16x2 {128 + (v & 15), 128 + ((v >> 16) & 15)}: (v & 0x000F000F) | 0x43004300
__device__ __forceinline__ uint32_t bf16x2_of_nibbles(uint32_t v) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(0x000F000Fu), "r"(0x43004300u));
    return r;
}

__device__ __forceinline__ void mma_bf16_m16n8k16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                  uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float half_bits_to_f32(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

struct Stage {
    uint4 qa, qb;                  // 32 codes of row q and of row q+8
    uint32_t sa, ma, sb, mb;       // fp16 bits of their scale and min
};

// Warp w of WARPS gets units [w*U/WARPS, (w+1)*U/WARPS).
__device__ __forceinline__ int range_begin(int w, int U, int warps) {
    return static_cast<int>((static_cast<int64_t>(w) * U) / warps);
}
// The warp whose range holds unit u.
__device__ __forceinline__ int range_owner(int u, int U, int warps) {
    return static_cast<int>(((static_cast<int64_t>(u) + 1) * warps - 1) / U);
}

// ------------------------------------------------------------------ the kernel
// MMA = true: per group, 8 mma.m16n8k16 (16 rows x 8 batch columns x 16 k) with
// fp32 accumulators.  MMA = false: the same sums on the CUDA cores, BT batch
// columns, fp32 FMA per code and column; both feed the same epilogue.
template <int WARPS, int DEPTH, bool MMA, int BT>
__global__ void __launch_bounds__(WARPS * 32, 1) q4_gemv_kernel(const GemvArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int t = lane & 3;    // 16-byte chunk of the 64-byte group row; k-slot quad
    const int q = lane >> 2;   // tile row (and row q + 8); batch column in the B fragment
    const int G = a.K >> 7;
    const int B = a.B;
    const int rb = blockIdx.x / a.k_splits;
    const int ks = blockIdx.x - rb * a.k_splits;
    const int r0 = static_cast<int>(static_cast<int64_t>(rb) * a.N / a.row_blocks);
    const int r1 = static_cast<int>(static_cast<int64_t>(rb + 1) * a.N / a.row_blocks);
    const int g0 = static_cast<int>(static_cast<int64_t>(ks) * G / a.k_splits);
    const int g1 = static_cast<int>(static_cast<int64_t>(ks + 1) * G / a.k_splits);
    const int Gs = g1 - g0;
    const int T = (r1 - r0 + 15) >> 4;
    const int U = T * Gs;
    const int ub = range_begin(warp, U, WARPS);
    const int ue = range_begin(warp + 1, U, WARPS);
    const size_t row_bytes = static_cast<size_t>(a.K) >> 1;

    // shared memory: x in B-fragment order | per-group x sums [Gs][8] | warp partials
    uint2* xs = reinterpret_cast<uint2*>(smem);
    float* ssum = reinterpret_cast<float*>(smem + static_cast<size_t>(Gs) * 256 * B);
    float* part = ssum + Gs * 8;

    if (a.l2_prefetch > 0 && threadIdx.x == 0 && a.k_splits == 1) {
        // the CTA's codes are one contiguous byte range: rows [r0, r1)
        const uint8_t* p = a.codes + static_cast<size_t>(r0) * row_bytes;
        size_t left = static_cast<size_t>(r1 - r0) * row_bytes;
        if (left > static_cast<size_t>(a.l2_prefetch)) left = static_cast<size_t>(a.l2_prefetch) & ~size_t(15);
        while (left > 0) {
            const uint32_t chunk = left > (1u << 20) ? (1u << 20) : static_cast<uint32_t>(left);
            prefetch_l2_bulk(p, chunk);
            p += chunk;
            left -= chunk;
        }
    }

    // ---- prologue: start streaming this warp's first DEPTH units (weights are read-only,
    // so this may run before the previous kernel in the stream has finished)
    Stage st[DEPTH];
    int lt = 0, lg = 0;  // load cursor: tile, local group
    if (ub < ue) { lt = ub / Gs; lg = ub - lt * Gs; }
    auto load_unit = [&](Stage& s) {
        const int ra = r0 + lt * 16 + q;
        const int rbw = ra + 8;
        const int g = g0 + lg;
        if (ra < r1) {
            s.qa = ld_stream_u4(a.codes + static_cast<size_t>(ra) * row_bytes + g * 64 + t * 16);
            s.sa = ld_nc_u16(a.scales + static_cast<size_t>(ra) * G + g);
            s.ma = ld_nc_u16(a.mins + static_cast<size_t>(ra) * G + g);
        } else {
            s.qa = make_uint4(0, 0, 0, 0); s.sa = 0; s.ma = 0;
        }
        if (rbw < r1) {
            s.qb = ld_stream_u4(a.codes + static_cast<size_t>(rbw) * row_bytes + g * 64 + t * 16);
            s.sb = ld_nc_u16(a.scales + static_cast<size_t>(rbw) * G + g);
            s.mb = ld_nc_u16(a.mins + static_cast<size_t>(rbw) * G + g);
        } else {
            s.qb = make_uint4(0, 0, 0, 0); s.sb = 0; s.mb = 0;
        }
        if (++lg == Gs) { lg = 0; ++lt; }
    };
#pragma unroll
    for (int d = 0; d < DEPTH; ++d)
        if (ub + d < ue) load_unit(st[d]);

    grid_dependency_wait();   // x may be the previous kernel's output; ws is shared with it
    allow_dependents();

    // ---- stage x in B-fragment order and the per-group sums of x
    {
        const int items = Gs * B * 16;  // (local group, column, chunk t, word i); (t, i) fastest
        const int iters = (items + blockDim.x - 1) / blockDim.x;
        for (int it = 0; it < iters; ++it) {
            const int idx = it * blockDim.x + threadIdx.x;
            float s = 0.f;
            const bool on = idx < items;
            int gl = 0, n = 0;
            if (on) {
                const int ti = idx & 15;
                const int gn = idx >> 4;
                n = gn % B;
                gl = gn / B;
                const int tt = ti >> 2, i = ti & 3;
                const uint4 v = *reinterpret_cast<const uint4*>(
                    a.x + static_cast<size_t>(n) * a.K + static_cast<size_t>(g0 + gl) * 128 + tt * 32 + i * 8);
                // v holds x[e0..e7] (two per word); fragment pairs are (e0,e4),(e1,e5) | (e2,e6),(e3,e7)
                uint2 p0, p1;
                p0.x = __byte_perm(v.x, v.z, 0x5410);
                p0.y = __byte_perm(v.x, v.z, 0x7632);
                p1.x = __byte_perm(v.y, v.w, 0x5410);
                p1.y = __byte_perm(v.y, v.w, 0x7632);
                const size_t base = static_cast<size_t>(gl * 4 + i) * 2 * (4 * B) + n * 4 + tt;
                xs[base] = p0;
                xs[base + 4 * B] = p1;
                s = bf16lo_to_f32(v.x);
                s += bf16hi_to_f32(v.x);
                s += bf16lo_to_f32(v.y);
                s += bf16hi_to_f32(v.y);
                s += bf16lo_to_f32(v.z);
                s += bf16hi_to_f32(v.z);
                s += bf16lo_to_f32(v.w);
                s += bf16hi_to_f32(v.w);
            }
            s += __shfl_xor_sync(0xffffffffu, s, 8);
            s += __shfl_xor_sync(0xffffffffu, s, 4);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            if (on && (idx & 15) == 0) ssum[gl * 8 + n] = s;
        }
        for (int idx = threadIdx.x; idx < Gs * 8; idx += blockDim.x)
            if ((idx & 7) >= B) ssum[idx] = 0.f;
    }
    __syncthreads();

    // ---- main loop over this warp's units
    float acc[4] = {0.f, 0.f, 0.f, 0.f};  // rows (q, q, q+8, q+8) x columns (2t, 2t+1, 2t, 2t+1)
    int ct = (ub < ue) ? ub / Gs : 0;     // compute cursor
    int cg = (ub < ue) ? ub - ct * Gs : 0;
    int seg = 0;
    const int first_tile = ct;
    const bool xon = q < B;

    auto flush = [&](int tile) {
        if (tile - first_tile >= a.smax) return;  // cannot happen with a plan from make_plan
        float* pp = part + static_cast<size_t>(warp * a.smax + (tile - first_tile)) * 16 * B;
        const int c0 = 2 * t, c1 = 2 * t + 1;
        if (c0 < B) { pp[q * B + c0] = acc[0]; pp[(q + 8) * B + c0] = acc[2]; }
        if (c1 < B) { pp[q * B + c1] = acc[1]; pp[(q + 8) * B + c1] = acc[3]; }
    };

    auto compute_unit = [&](const Stage& s) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t wa[4] = {s.qa.x, s.qa.y, s.qa.z, s.qa.w};
        const uint32_t wb[4] = {s.qb.x, s.qb.y, s.qb.z, s.qb.w};
        const uint2* xg = xs + static_cast<size_t>(cg) * 8 * (4 * B);
        if constexpr (MMA) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t a0 = bf16x2_of_nibbles(wa[i]);
                const uint32_t a1 = bf16x2_of_nibbles(wa[i] >> 4);
                const uint32_t a2 = bf16x2_of_nibbles(wa[i] >> 8);
                const uint32_t a3 = bf16x2_of_nibbles(wa[i] >> 12);
                const uint32_t b0 = bf16x2_of_nibbles(wb[i]);
                const uint32_t b1 = bf16x2_of_nibbles(wb[i] >> 4);
                const uint32_t b2 = bf16x2_of_nibbles(wb[i] >> 8);
                const uint32_t b3 = bf16x2_of_nibbles(wb[i] >> 12);
                uint2 x0 = make_uint2(0, 0), x1 = make_uint2(0, 0);
                if (xon) {
                    x0 = xg[(i * 2 + 0) * (4 * B) + lane];
                    x1 = xg[(i * 2 + 1) * (4 * B) + lane];
                }
                mma_bf16_m16n8k16(c, a0, b0, a1, b1, x0.x, x0.y);
                mma_bf16_m16n8k16(c, a2, b2, a3, b3, x1.x, x1.y);
            }
        } else {
            float pa[BT], pb[BT];
#pragma unroll
            for (int n = 0; n < BT; ++n) { pa[n] = 0.f; pb[n] = 0.f; }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const uint32_t A0 = bf16x2_of_nibbles(wa[i] >> (8 * p));
                    const uint32_t A1 = bf16x2_of_nibbles(wa[i] >> (8 * p + 4));
                    const uint32_t B0 = bf16x2_of_nibbles(wb[i] >> (8 * p));
                    const uint32_t B1 = bf16x2_of_nibbles(wb[i] >> (8 * p + 4));
                    const float a00 = bf16lo_to_f32(A0), a01 = bf16hi_to_f32(A0);
                    const float a10 = bf16lo_to_f32(A1), a11 = bf16hi_to_f32(A1);
                    const float b00 = bf16lo_to_f32(B0), b01 = bf16hi_to_f32(B0);
                    const float b10 = bf16lo_to_f32(B1), b11 = bf16hi_to_f32(B1);
#pragma unroll
                    for (int n = 0; n < BT; ++n) {
                        uint2 xv = make_uint2(0, 0);
                        if (n < B) xv = xg[(i * 2 + p) * (4 * B) + n * 4 + t];
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
            // sum over the quad's four 32-column chunks; every lane of the quad gets the same value
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
        const float2 S = *reinterpret_cast<const float2*>(ssum + cg * 8 + 2 * t);
        const float sa = half_bits_to_f32(s.sa), ma = half_bits_to_f32(s.ma);
        const float sb = half_bits_to_f32(s.sb), mb = half_bits_to_f32(s.mb);
        const float ma2 = fmaf(-128.f, sa, ma);
        const float mb2 = fmaf(-128.f, sb, mb);
        acc[0] = fmaf(sa, c[0], acc[0]);
        acc[0] = fmaf(ma2, S.x, acc[0]);
        acc[1] = fmaf(sa, c[1], acc[1]);
        acc[1] = fmaf(ma2, S.y, acc[1]);
        acc[2] = fmaf(sb, c[2], acc[2]);
        acc[2] = fmaf(mb2, S.x, acc[2]);
        acc[3] = fmaf(sb, c[3], acc[3]);
        acc[3] = fmaf(mb2, S.y, acc[3]);
        if (++cg == Gs) {
            flush(ct);
            acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
            cg = 0;
            ++ct;
        }
    };

    for (int u = ub; u < ue; u += DEPTH) {
#pragma unroll
        for (int d = 0; d < DEPTH; ++d) {
            if (u + d < ue) {
                const Stage cur = st[d];
                if (u + d + DEPTH < ue) load_unit(st[d]);
                compute_unit(cur);
            }
        }
    }
    if (ub < ue && cg != 0) flush(ct);  // range ended inside a tile
    (void)seg;
    __syncthreads();

    // ---- add the warp partials of each tile in warp order
    const int rows = r1 - r0;
    const bool split = a.k_splits > 1;
    for (int idx = threadIdx.x; idx < rows * B; idx += blockDim.x) {
        const int b = idx / rows;
        const int rr = idx - b * rows;
        const int j = rr >> 4, rl = rr & 15;
        const int wf = range_owner(j * Gs, U, WARPS);
        const int wl = range_owner(j * Gs + Gs - 1, U, WARPS);
        float sum = 0.f;
        for (int w = wf; w <= wl; ++w) {
            const int bw = range_begin(w, U, WARPS);
            if (bw >= range_begin(w + 1, U, WARPS)) continue;  // empty range
            const int sgi = j - bw / Gs;
            sum += part[(static_cast<size_t>(w * a.smax + sgi) * 16 + rl) * B + b];
        }
        if (!split)
            a.y[static_cast<size_t>(b) * a.N + r0 + rr] = sum;
        else
            a.ws_part[(static_cast<size_t>(ks) * B + b) * a.N + r0 + rr] = sum;
    }
    if (!split) return;

    // ---- k-split: the last CTA of this row block adds the partials in k-split order
    __shared__ int is_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned prev = atomicAdd(a.ws_cnt + rb, 1u);
        is_last = (prev == static_cast<unsigned>(a.k_splits - 1));
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    for (int idx = threadIdx.x; idx < rows * B; idx += blockDim.x) {
        const int b = idx / rows;
        const int rr = idx - b * rows;
        float sum = 0.f;
        for (int k2 = 0; k2 < a.k_splits; ++k2)
            sum += __ldcg(a.ws_part + (static_cast<size_t>(k2) * B + b) * a.N + r0 + rr);
        a.y[static_cast<size_t>(b) * a.N + r0 + rr] = sum;
    }
    if (threadIdx.x == 0) a.ws_cnt[rb] = 0u;  // ready for the next call
}

// ------------------------------------------------------------------ argmax
__device__ __forceinline__ bool ranks_above(float v, int i, float bv, int bi) {
    const bool vn = v != v, bn = bv != bv;
    if (vn || bn) return vn && (!bn || i < bi);
    return v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(1024) q4_argmax_kernel(const float* __restrict__ Y, int N, int32_t* idx) {
    grid_dependency_wait();  // Y is usually the previous kernel's output
    const float* row = Y + static_cast<size_t>(blockIdx.x) * N;
    float bv = -__int_as_float(0x7f800000);
    int bi = 0x7fffffff;
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
        const float v = __ldg(row + i);
        if (ranks_above(v, i, bv, bi)) { bv = v; bi = i; }
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

// ------------------------------------------------------------------ host: plan
struct Plan {
    int row_blocks, k_splits, warps, depth, smax, kernel, sms, l2_prefetch;
    bool pdl;
    int Gs_max;
};

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

size_t plan_smem(const Plan& p, int B) {
    return static_cast<size_t>(p.Gs_max) * 256 * B + static_cast<size_t>(p.Gs_max) * 32 +
           static_cast<size_t>(p.warps) * p.smax * 16 * B * 4;
}

// The split depends on (N, K, SM count) and on benchmarking overrides only.
bool make_plan(int64_t N, int64_t K, int sms, Plan* out) {
    Plan p{};
    const int G = static_cast<int>(K / 128);
    p.sms = sms;
    p.kernel = env_int("Q4_KERNEL", 0) == 1 ? 1 : 0;
    p.warps = env_int("Q4_WARPS", 16);
    p.depth = env_int("Q4_DEPTH", 4);
    if (p.kernel == 1) p.depth = 4;
    const bool ok_shape = (p.warps == 16 && (p.depth == 2 || p.depth == 4 || p.depth == 6)) ||
                          (p.warps == 8 && (p.depth == 4 || p.depth == 8)) ||
                          (p.warps == 32 && p.depth == 2);
    if (!ok_shape || (p.kernel == 1 && p.warps != 16)) { p.warps = 16; p.depth = 4; }
    p.pdl = env_int("Q4_PDL", 1) != 0;
    p.l2_prefetch = env_int("Q4_L2_PREFETCH", 0);
    // x for 8 columns of a k-slice takes 16 bytes per column of K in shared memory
    int ks = static_cast<int>((K + 8191) / 8192);
    const int ks_env = env_int("Q4_KSPLIT", 0);
    if (ks_env > 0) ks = ks_env;
    if (ks > G) ks = G;
    if (ks < 1) ks = 1;
    for (;; ++ks) {
        int rb_max = sms / ks;
        if (rb_max < 1) rb_max = 1;
        const int64_t tiles = (N + 15) / 16;
        p.row_blocks = static_cast<int>(tiles < rb_max ? tiles : rb_max);
        p.k_splits = ks;
        const int64_t rows_max = (N + p.row_blocks - 1) / p.row_blocks;
        const int Tm = static_cast<int>((rows_max + 15) / 16);
        const int gs_min = G / ks;
        p.Gs_max = (G + ks - 1) / ks;
        const int64_t Um = static_cast<int64_t>(Tm) * p.Gs_max;
        const int upw = static_cast<int>((Um + p.warps - 1) / p.warps);
        int smax = (upw + gs_min - 1) / gs_min + 1;
        if (smax > Tm) smax = Tm;
        if (smax < 1) smax = 1;
        p.smax = smax;
        if (plan_smem(p, kMaxB) <= kSmemLimit) break;
        if (ks >= G) return false;
    }
    *out = p;
    return true;
}

size_t plan_ws_bytes(const Plan& p, int64_t N, int B) {
    if (p.k_splits <= 1) return 0;
    const size_t cnt = (static_cast<size_t>(p.row_blocks) * 4 + 255) / 256 * 256;
    return cnt + static_cast<size_t>(p.k_splits) * B * N * 4;
}

using KernelFn = void (*)(GemvArgs);

KernelFn pick_kernel(const Plan& p, int B) {
    if (p.kernel == 1) {
        if (B <= 1) return q4_gemv_kernel<16, 4, false, 1>;
        if (B <= 2) return q4_gemv_kernel<16, 4, false, 2>;
        if (B <= 4) return q4_gemv_kernel<16, 4, false, 4>;
        return q4_gemv_kernel<16, 4, false, 8>;
    }
    if (p.warps == 8) return p.depth == 8 ? q4_gemv_kernel<8, 8, true, 8> : q4_gemv_kernel<8, 4, true, 8>;
    if (p.warps == 32) return q4_gemv_kernel<32, 2, true, 8>;
    if (p.depth == 2) return q4_gemv_kernel<16, 2, true, 8>;
    if (p.depth == 6) return q4_gemv_kernel<16, 6, true, 8>;
    return q4_gemv_kernel<16, 4, true, 8>;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

q4_status check_matrix(const q4_matrix* W) {
    if (!W || !W->codes || !W->scales || !W->mins) return Q4_ERR_INVALID_ARG;
    if (W->N <= 0) return Q4_ERR_INVALID_ARG;
    if (W->N > 0x7fffffffLL) return Q4_ERR_UNSUPPORTED_SHAPE;
    if (W->K <= 0 || W->K % 128 != 0 || W->K > kMaxK) return Q4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(W->codes, 16) || !aligned(W->scales, 2) || !aligned(W->mins, 2)) return Q4_ERR_MISALIGNED;
    return Q4_OK;
}

q4_status check_io(const uint16_t* X, int B, const float* Y) {
    if (!X || !Y) return Q4_ERR_INVALID_ARG;
    if (B < 1 || B > kMaxB) return Q4_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(Y, 4)) return Q4_ERR_MISALIGNED;
    return Q4_OK;
}

bool fault_injected() {
    const char* v = std::getenv("Q4_FAULT_INJECT");
    return v && std::strcmp(v, "launch") == 0;
}

bool smem_attr_set(KernelFn fn, int dev) {
    // cudaFuncSetAttribute once per (kernel, device)
    struct Entry { KernelFn fn; int dev; };
    static Entry done[256];
    static int n_done = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_done; ++i)
        if (done[i].fn == fn && done[i].dev == dev) return true;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemLimit)) !=
        cudaSuccess)
        return false;
    if (n_done < 256) done[n_done++] = Entry{fn, dev};
    return true;
}

q4_status launch_gemv(const q4_matrix* W, const uint16_t* X, int B, float* Y, void* ws, const Plan& p,
                      int dev, cudaStream_t stream) {
    GemvArgs a{};
    a.codes = W->codes;
    a.scales = W->scales;
    a.mins = W->mins;
    a.x = X;
    a.y = Y;
    a.N = static_cast<int>(W->N);
    a.K = static_cast<int>(W->K);
    a.B = B;
    a.row_blocks = p.row_blocks;
    a.k_splits = p.k_splits;
    a.smax = p.smax;
    a.l2_prefetch = p.l2_prefetch;
    if (p.k_splits > 1) {
        const size_t cnt = (static_cast<size_t>(p.row_blocks) * 4 + 255) / 256 * 256;
        a.ws_cnt = static_cast<unsigned int*>(ws);
        a.ws_part = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + cnt);
    }
    if (fault_injected()) return Q4_ERR_CUDA;
    KernelFn fn = pick_kernel(p, B);
    if (!smem_attr_set(fn, dev)) return Q4_ERR_CUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(p.row_blocks * p.k_splits));
    cfg.blockDim = dim3(static_cast<unsigned>(p.warps * 32));
    cfg.dynamicSmemBytes = plan_smem(p, B);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = p.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, a) == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

}  // namespace

// ------------------------------------------------------------------ C ABI
extern "C" size_t q4_workspace_bytes(int64_t N, int64_t K, int B) {
    if (N <= 0 || N > 0x7fffffffLL || K <= 0 || K % 128 || K > kMaxK || B < 1 || B > kMaxB) return 0;
    const int sms = device_sm_count(nullptr);
    if (sms <= 0) return 0;
    Plan p;
    if (!make_plan(N, K, sms, &p)) return 0;
    return plan_ws_bytes(p, N, B);
}

extern "C" q4_status q4_plan(int64_t N, int64_t K, q4_plan_info* out) {
    if (!out || N <= 0) return Q4_ERR_INVALID_ARG;
    if (N > 0x7fffffffLL || K <= 0 || K % 128 || K > kMaxK) return Q4_ERR_UNSUPPORTED_SHAPE;
    const int sms = device_sm_count(nullptr);
    if (sms <= 0) return Q4_ERR_CUDA;
    Plan p;
    if (!make_plan(N, K, sms, &p)) return Q4_ERR_UNSUPPORTED_SHAPE;
    out->row_blocks = p.row_blocks;
    out->k_splits = p.k_splits;
    out->warps_per_cta = p.warps;
    out->prefetch_depth = p.depth;
    out->kernel = p.kernel;
    out->sm_count = p.sms;
    return Q4_OK;
}

extern "C" q4_status q4_gemm_skinny(const q4_matrix* W, const uint16_t* X, int B, float* Y, void* ws,
                                    size_t ws_bytes, void* stream) {
    q4_status s = check_matrix(W);
    if (s != Q4_OK) return s;
    if ((s = check_io(X, B, Y)) != Q4_OK) return s;
    int dev = 0;
    const int sms = device_sm_count(&dev);
    if (sms <= 0) return Q4_ERR_CUDA;
    Plan p;
    if (!make_plan(W->N, W->K, sms, &p)) return Q4_ERR_UNSUPPORTED_SHAPE;
    const size_t need = plan_ws_bytes(p, W->N, B);
    if (need > 0) {
        if (!ws || ws_bytes < need) return Q4_ERR_WORKSPACE;
        if (!aligned(ws, 16)) return Q4_ERR_MISALIGNED;
    }
    return launch_gemv(W, X, B, Y, ws, p, dev, static_cast<cudaStream_t>(stream));
}

extern "C" q4_status q4_gemv(const q4_matrix* W, const uint16_t* x, float* y, void* ws, size_t ws_bytes,
                             void* stream) {
    return q4_gemm_skinny(W, x, 1, y, ws, ws_bytes, stream);
}

extern "C" q4_status q4_decode_step(const q4_matrix* mats, int n_mats, const uint16_t* const* X,
                                    float* const* Y, int B, void* ws, size_t ws_bytes, void* stream) {
    if (!mats || !X || !Y || n_mats < 1) return Q4_ERR_INVALID_ARG;
    if (B < 1 || B > kMaxB) return Q4_ERR_INVALID_ARG;
    int dev = 0;
    const int sms = device_sm_count(&dev);
    if (sms <= 0) return Q4_ERR_CUDA;
    size_t need = 0;
    for (int i = 0; i < n_mats; ++i) {
        q4_status s = check_matrix(&mats[i]);
        if (s != Q4_OK) return s;
        if ((s = check_io(X[i], B, Y[i])) != Q4_OK) return s;
        Plan p;
        if (!make_plan(mats[i].N, mats[i].K, sms, &p)) return Q4_ERR_UNSUPPORTED_SHAPE;
        const size_t n = plan_ws_bytes(p, mats[i].N, B);
        if (n > need) need = n;
    }
    if (need > 0) {
        if (!ws || ws_bytes < need) return Q4_ERR_WORKSPACE;
        if (!aligned(ws, 16)) return Q4_ERR_MISALIGNED;
    }
    for (int i = 0; i < n_mats; ++i) {
        Plan p;
        make_plan(mats[i].N, mats[i].K, sms, &p);
        const q4_status s = launch_gemv(&mats[i], X[i], B, Y[i], ws, p, dev, static_cast<cudaStream_t>(stream));
        if (s != Q4_OK) return s;
    }
    return Q4_OK;
}

extern "C" q4_status q4_argmax_f32(const float* Y, int B, int64_t N, int32_t* idx, void* stream) {
    if (!Y || !idx || B < 1 || B > kMaxB || N < 1 || N > 0x7fffffffLL) return Q4_ERR_INVALID_ARG;
    if (!aligned(Y, 4) || !aligned(idx, 4)) return Q4_ERR_MISALIGNED;
    if (fault_injected()) return Q4_ERR_CUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(B));
    cfg.blockDim = dim3(1024);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = env_int("Q4_PDL", 1) != 0 ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, q4_argmax_kernel, Y, static_cast<int>(N), idx) == cudaSuccess ? Q4_OK
                                                                                                : Q4_ERR_CUDA;
}
