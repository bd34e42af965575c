// Flash-decoding for GB300 (sm_103a): one decode step of grouped-query attention over a KV cache.
//
// What is computed (rumik-oss-1 int4 engine page, rtts.neoandmatrix.me, "Step 6: flash-decoding
// for long clips"):
//     O[b, h, :] = sum_{p < len[b]} softmax_p(scale * <Q[b,h,:], K[b,h/g,p,:]>) V[b,h/g,p,:]
// with g = Hq / Hkv query heads per KV head.  As on the page, each KV head's cache is cut into
// pieces (chunks) processed in parallel, the g grouped query heads are the rows of one
// matrix-multiply tile, and a separate small kernel merges the per-chunk results.
//
// Chunking: chunk length cs = max(ceil(len / C) rounded up to 16, a minimum length), C chunks
// per KV head at most.  It depends on len[b], C and the minimum and nothing else (never on B).
//
// Split kernel: CTAs (x, KV head, sequence b) of four independent warps.  The warps of one
// (b, KV head) take its chunks in turn (warp w: chunks w, w + nw, ...) and one warp computes a
// whole chunk: the chunk's partial result (m, l, o) stays in the warp's registers and goes to
// the workspace when the chunk ends.  A chunk's arithmetic is the same whichever warp runs it,
// so the host may choose the number of CTAs per KV head from B and the SM count without
// changing a bit of any sequence's result.  A warp streams the 16-position tiles of its chunks
// -- keys and values, every byte once -- through its own ring of three shared-memory slots, two
// tiles ahead, across chunk boundaries: each lane issues one bulk copy (the TMA engine) of one
// key or value row into a padded slot row, and an mbarrier per slot counts the bytes in.  (A
// second fill, 16-byte cp.async copies that each lane reads back itself, streams measurably
// slower and is kept as an option.)  Per tile it
//   * computes the 16 x 16 score tile S = Q K^T with mma.m16n8k16 (rows: the g query heads of
//     this KV head, padded to 16 with zero queries; columns: positions), bf16 in, fp32 out;
//   * updates a running softmax in base 2 (u = s * scale * log2 e; running maximum m and sum l
//     per row; p = 2^(u - m); the sums are rescaled only when a row's maximum grows);
//   * adds P V with mma.m16n8k16.  P is split into bf16 parts hi + lo (|p - hi - lo| <= 2^-18 p),
//     two products per tile, so the weights keep fp32-class precision on bf16 tensor cores.
// A dot product does not depend on the order of its terms, so each lane's fragments are taken
// in the order its 16-byte copies deliver them: the query fragments follow the same permutation
// of the head dimension as the keys.  The partial o is stored in the accumulator's own order
// (see fd_dim) and mapped back to head dimensions by the combine kernel.
//
// Combine kernel: one CTA per (query head, sequence), 512 threads (256 when the pairs exceed one
// wave of SMs):   O = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c,   M = max_c m_c.
// The chunks fall into 512/D classes (chunk index modulo 512/D); each class is summed in chunk
// order and the classes in class order, for the outputs and the denominator alike, so the bits do
// not depend on the thread count.  The first round of partials (48 per thread) and all chunks'
// (m, l) are loaded together with the sequence's length, bounded by the chunk capacity: one
// memory round trip for up to 192 chunks (D = 128, 512 threads) before the arithmetic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <utility>

#include "q4.h"
#include "q4_common.cuh"

namespace {

constexpr int kFdWarps = 4;
constexpr int kFdStages = 3;           // ring slots per warp: two tiles in flight while one is used
constexpr int kFdMaxGroup = 16;        // query heads per KV head: one 16-row tensor-core tile
constexpr int kFdMaxChunks = 4096;
constexpr int kFdMinChunk = 32;        // positions: at least two tiles per chunk
constexpr int64_t kFdMaxLen = 1 << 30;

struct FdParams {
    const uint16_t* Q;        // [B, Hq, D] bf16
    const uint16_t* K;        // [B, Hkv, Lmax, D] bf16
    const uint16_t* V;        // [B, Hkv, Lmax, D] bf16
    const int32_t* lengths;   // [B]
    float* O;                 // [B, Hq, D]
    float* part;              // [B, Hkv, C, g, D]  chunk partial sums o, accumulator order
    float* ml;                // [B, Hkv, C, g, 2]  chunk partial (m, l)
    int64_t Lmax;
    float c;                  // scale * log2(e)
    int Hkv, g, C, min_chunk;
};

constexpr uint32_t kFdWaitLimit = 1u << 22;  // mbarrier polls before a wait gives up

__device__ unsigned int g_fd_device_error;  // set when a bounded wait gives up

// Per-warp ring slot of one 16-position tile.  Bulk slots pad the rows (keys to 2D + 64 bytes,
// values to 2D + 16) so that the lanes' 16-byte fragment reads fall in distinct bank groups.
template <int D, bool BULK>
struct FdSlot {
    static constexpr int kKeyStride = 2 * D + 64;
    static constexpr int kValueStride = 2 * D + 16;
    static constexpr int kBytes = BULK ? 16 * (kKeyStride + kValueStride) : 16 * 2 * D * 2;
};

__device__ __forceinline__ uint4 lds_u4(const unsigned char* p) { return *reinterpret_cast<const uint4*>(p); }

// attended positions of sequence b (clamped to 0..Lmax), its chunk length and chunk count
__device__ __forceinline__ void fd_chunking(const FdParams& p, int b, int& len, int& cs, int& used) {
    int64_t n = static_cast<int32_t>(ld_dep_u32(p.lengths + b));
    n = n < 0 ? 0 : (n > p.Lmax ? p.Lmax : n);
    const int64_t per = (n + p.C - 1) / p.C;
    int64_t c = (per + 15) / 16 * 16;
    if (c < p.min_chunk) c = p.min_chunk;
    len = static_cast<int>(n);
    cs = static_cast<int>(c);
    used = static_cast<int>((n + c - 1) / c);  // <= C
}

// head dimension of entry e of a stored partial: the P V accumulator of column tile n holds
// lane t's columns 2t, 2t+1, i.e. dims 64(n/8) + 8(2t + k) + n%8, stored at e = 8n + 2t + k
__device__ __forceinline__ int fd_dim(int e) {
    const int n = e >> 3, t = (e >> 1) & 3, k = e & 1;
    return 64 * (n >> 3) + 8 * (2 * t + k) + (n & 7);
}

// 2^x with the hardware's approximate base-2 exponential (relative error about 2^-22; results
// below 2^-126 flush to 0; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// p = hi + lo: hi = bf16(p) per element, lo = bf16(p - hi)
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = bf16x2_bits(a - __low2float(h), b - __high2float(h));
}

template <int D, int S, bool BULK>
__global__ void __launch_bounds__(kFdWarps * 32) q4_flash_split_kernel(const __grid_constant__ FdParams p) {
    constexpr int KJ = D / 32;  // 16-byte key pieces per position per lane (4 lanes share a key)
    constexpr int VJ = D / 64;  // 16-byte value pieces per position per lane (8 lanes share a row)
    constexpr int NP = D / 8;   // pieces per lane per tile: 2 KJ keys + 4 VJ values
    constexpr int NT = D / 8;   // output column tiles of P V
    constexpr int KS = D / 16;  // k-steps of Q K^T
    constexpr int KSTR = FdSlot<D, BULK>::kKeyStride, VSTR = FdSlot<D, BULK>::kValueStride;
    constexpr int SLOT = FdSlot<D, BULK>::kBytes;
    // [warp][slot]: cp.async slots hold [piece][lane] (each lane reads back only what it copied);
    // bulk slots hold 16 padded key rows then 16 padded value rows, then the slots' mbarriers
    extern __shared__ __align__(16) unsigned char fd_smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int q = lane >> 2, t = lane & 3;
    const int kvh = blockIdx.y, b = blockIdx.z;
    const int g = p.g;

    grid_dependency_wait();  // queries and cache come from the kernels before
    allow_dependents();

    int len, cs, used;
    fd_chunking(p, b, len, cs, used);
    const int w0 = blockIdx.x * kFdWarps + warp, nw = gridDim.x * kFdWarps;
    if (w0 >= used) return;  // the warps are independent: no block-wide synchronisation below

    const size_t head = static_cast<size_t>(b) * p.Hkv + kvh;
    const uint16_t* Kh = p.K + head * p.Lmax * D;
    const uint16_t* Vh = p.V + head * p.Lmax * D;
    uint4* ring = reinterpret_cast<uint4*>(fd_smem_raw) + static_cast<size_t>(warp) * S * NP * 32 + lane;
    unsigned char* wslots = fd_smem_raw + static_cast<size_t>(warp) * S * SLOT;
    uint64_t* bars = reinterpret_cast<uint64_t*>(fd_smem_raw + static_cast<size_t>(kFdWarps) * S * SLOT) + warp * S;
    if constexpr (BULK) {
        if (lane == 0) {
#pragma unroll
            for (int sl = 0; sl < S; ++sl) mbar_init(&bars[sl], 1);
            fence_barrier_init();
        }
        __syncwarp();
    }

    // The warp's tiles in order: chunk w0's, then chunk w0 + nw's, ...  Copy the next one into
    // the next slot: keys of positions base + 8h + q (h = 0, 1), dims 32j + 8t .. +7; values of
    // positions base + 8(i/2) + 2t + i%2, dims 64j + 8q .. +7.  Positions past the chunk's end
    // copy its last row (finite data; their weight is exactly 0).  One commit group per call.
    int ic = w0, it = 0, islot = 0;
    auto issue_next = [&]() {
        if constexpr (BULK) __syncwarp();  // every lane has read the slot being refilled
        if (ic < used) {
            const int s0 = ic * cs, e0 = min(len, s0 + cs);
            const int base = s0 + 16 * it;
            if constexpr (BULK) {
                // lane r < 16: key row base + r; lane 16 + r: value row base + r (one bulk copy each)
                unsigned char* dst = wslots + static_cast<size_t>(islot) * SLOT;
                if (lane == 0) mbar_arrive_expect_tx(&bars[islot], 32 * 2 * D);
                __syncwarp();
                const int r = lane & 15, pos = min(base + r, e0 - 1);
                if (lane < 16)
                    bulk_g2s(dst + r * KSTR, Kh + static_cast<size_t>(pos) * D, 2 * D, &bars[islot]);
                else
                    bulk_g2s(dst + 16 * KSTR + r * VSTR, Vh + static_cast<size_t>(pos) * D, 2 * D, &bars[islot]);
            } else {
            uint4* dst = ring + static_cast<size_t>(islot) * NP * 32;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int pos = min(base + 8 * h + q, e0 - 1);
#pragma unroll
                for (int j = 0; j < KJ; ++j)
                    cp_async16(dst + (h * KJ + j) * 32, Kh + static_cast<size_t>(pos) * D + 32 * j + 8 * t);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int pos = min(base + 8 * (i >> 1) + 2 * t + (i & 1), e0 - 1);
#pragma unroll
                for (int j = 0; j < VJ; ++j)
                    cp_async16(dst + (2 * KJ + i * VJ + j) * 32, Vh + static_cast<size_t>(pos) * D + 64 * j + 8 * q);
            }
            }
            if (base + 16 >= e0) {  // that was the chunk's last tile
                ic += nw;
                it = 0;
            } else {
                ++it;
            }
        }
        if constexpr (!BULK) cp_async_commit();
        islot = islot == S - 1 ? 0 : islot + 1;
    };
#pragma unroll
    for (int sl = 0; sl < S - 1; ++sl) issue_next();

    // A operand of Q K^T: rows q and q+8 = query heads kvh*g + row (zero rows past g).  k-step m
    // covers head-dimension slots {2t, 2t+1} -> d0, d0+1 and {2t+8, 2t+9} -> d0+2, d0+3 with
    // d0 = 32 (m/2) + 8t + 4 (m%2), the order in which this lane's key pieces arrive.
    const uint16_t* Qh = p.Q + head * g * D;
    uint32_t qa[KS][4];
#pragma unroll
    for (int m = 0; m < KS; ++m) {
        const int d0 = 32 * (m >> 1) + 8 * t + 4 * (m & 1);
        const uint2 r0 = q < g ? ld_dep_u2(Qh + q * D + d0) : make_uint2(0u, 0u);
        const uint2 r1 = q + 8 < g ? ld_dep_u2(Qh + (q + 8) * D + d0) : make_uint2(0u, 0u);
        qa[m][0] = r0.x;
        qa[m][1] = r1.x;
        qa[m][2] = r0.y;
        qa[m][3] = r1.y;
    }

    int rs = 0;           // ring slot of the tile being computed
    uint32_t phase = 0;   // bulk: parity of that slot's current use (flips after slot S-1)
    bool ok = true;
    for (int cc = w0; cc < used && ok; cc += nw) {
        const int s0 = cc * cs, e0 = min(len, s0 + cs);
        float acc[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        float mrow[2] = {-INFINITY, -INFINITY};  // rows q, q+8 (the same in the 4 lanes of a quad)
        float lsum[2] = {0.f, 0.f};              // this lane's share of the row sums

        for (int base = s0; base < e0; base += 16) {
            uint4 kr[2][KJ], vr[4][VJ];
            if constexpr (BULK) {
                if (!mbar_wait(&bars[rs], phase, kFdWaitLimit)) {  // the tile's 32 rows have landed
                    ok = false;
                    break;
                }
                const unsigned char* src = wslots + static_cast<size_t>(rs) * SLOT;
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int j = 0; j < KJ; ++j) kr[h][j] = lds_u4(src + (8 * h + q) * KSTR + 64 * j + 16 * t);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < VJ; ++j)
                        vr[i][j] = lds_u4(src + 16 * KSTR + (8 * (i >> 1) + 2 * t + (i & 1)) * VSTR + 128 * j + 16 * q);
                issue_next();
            } else {
                cp_async_wait<S - 2>();  // this lane's copies of the tile have landed
                issue_next();
                const uint4* src = ring + static_cast<size_t>(rs) * NP * 32;
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int j = 0; j < KJ; ++j) kr[h][j] = src[(h * KJ + j) * 32];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < VJ; ++j) vr[i][j] = src[(2 * KJ + i * VJ + j) * 32];
            }
            if (rs == S - 1) {
                rs = 0;
                phase ^= 1u;
            } else {
                ++rs;
            }

            // S: s[h][0..1] = row q, columns 2t, 2t+1 of half h; s[h][2..3] = row q+8.  Even and
            // odd k-steps go to separate accumulators (four independent chains), added at the end.
            float s[2][4], s2[2][4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int m = 0; m < KS; ++m) {
                    const uint4& kv = kr[h][m >> 1];
                    float (&d)[4] = (m & 1) ? s2[h] : s[h];
                    const uint32_t b0 = (m & 1) ? kv.z : kv.x, b1 = (m & 1) ? kv.w : kv.y;
                    if (m < 2)
                        mma_bf16_m16n8k16_zc(d, qa[m][0], qa[m][1], qa[m][2], qa[m][3], b0, b1);
                    else
                        mma_bf16_m16n8k16(d, qa[m][0], qa[m][1], qa[m][2], qa[m][3], b0, b1);
                }
            }

            // online softmax in base 2; the tile's first position is always valid, so the new
            // maximum is finite.  Only a chunk's last tile can hold positions past its end.
            float tmax[2] = {-INFINITY, -INFINITY};
            const bool tail = base + 16 > e0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float u = (s[h][e] + s2[h][e]) * p.c;
                    if (tail && base + 8 * h + 2 * t + (e & 1) >= e0) u = -INFINITY;
                    s[h][e] = u;
                    tmax[e >> 1] = fmaxf(tmax[e >> 1], u);
                }
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 1));
                tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 2));
            }
            // a row whose maximum grew rescales its sums by 2^(m_old - m_new) (0 on the chunk's
            // first tile); otherwise the factor would be exactly 1 and the warp skips the step
            if (__any_sync(0xffffffffu, tmax[0] > mrow[0] || tmax[1] > mrow[1])) {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float mn = fmaxf(mrow[r], tmax[r]);
                    const float alpha = ex2(mrow[r] - mn);
                    mrow[r] = mn;
                    lsum[r] *= alpha;
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        acc[n][2 * r] *= alpha;
                        acc[n][2 * r + 1] *= alpha;
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float pe = ex2(s[h][e] - mrow[e >> 1]);
                    s[h][e] = pe;
                    lsum[e >> 1] += pe;
                }
            }

            // A operand of P V: slots 0..7 = half 0's positions, 8..15 = half 1's
            uint32_t ph[4], pl[4];
            split_bf16x2(s[0][0], s[0][1], ph[0], pl[0]);
            split_bf16x2(s[0][2], s[0][3], ph[1], pl[1]);
            split_bf16x2(s[1][0], s[1][1], ph[2], pl[2]);
            split_bf16x2(s[1][2], s[1][3], ph[3], pl[3]);
            // B operand for column tile n: lane column q <-> dim 64(n/8) + 8q + n%8; k slots
            // 2t, 2t+1 <-> values vr[0], vr[1]; slots 2t+8, 2t+9 <-> vr[2], vr[3]
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int j = n >> 3, w = (n & 7) >> 1;
                const uint32_t sel = (n & 1) ? 0x7632u : 0x5410u;
                const uint32_t* v0 = reinterpret_cast<const uint32_t*>(&vr[0][j]);
                const uint32_t* v1 = reinterpret_cast<const uint32_t*>(&vr[1][j]);
                const uint32_t* v2 = reinterpret_cast<const uint32_t*>(&vr[2][j]);
                const uint32_t* v3 = reinterpret_cast<const uint32_t*>(&vr[3][j]);
                const uint32_t b0 = __byte_perm(v0[w], v1[w], sel);
                const uint32_t b1 = __byte_perm(v2[w], v3[w], sel);
                mma_bf16_m16n8k16(acc[n], ph[0], ph[1], ph[2], ph[3], b0, b1);
                mma_bf16_m16n8k16(acc[n], pl[0], pl[1], pl[2], pl[3], b0, b1);
            }
        }

        // the chunk's partial: row sums over the quad; o of rows < g in accumulator order
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            lsum[r] += __shfl_xor_sync(0xffffffffu, lsum[r], 1);
            lsum[r] += __shfl_xor_sync(0xffffffffu, lsum[r], 2);
        }
        const size_t slot = (head * p.C + cc) * g;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int row = q + 8 * r;
            if (row < g) {
                float2* o = reinterpret_cast<float2*>(p.part + (slot + row) * D);
#pragma unroll
                for (int n = 0; n < NT; ++n) o[4 * n + t] = make_float2(acc[n][2 * r], acc[n][2 * r + 1]);
                if (t == 0) *reinterpret_cast<float2*>(p.ml + (slot + row) * 2) = make_float2(mrow[r], lsum[r]);
            }
        }
    }
    if constexpr (BULK) {
        if (!ok) {
            // a copy did not land within the limit: report it, give every slot a bounded last wait
            // so that no copy is left writing into this block's shared memory, and stop
            if (lane == 0) atomicOr(&g_fd_device_error, 1u);
#pragma unroll
            for (int sl = 0; sl < S; ++sl) {
                mbar_wait(&bars[sl], 0u, kFdWaitLimit);
                mbar_wait(&bars[sl], 1u, kFdWaitLimit);
            }
        }
    } else {
        cp_async_wait<0>();
    }
}

// fixed-order block reductions over NT threads (the same tree for every call)
template <bool MAX, int NT>
__device__ __forceinline__ float block_reduce(float v, float* red) {
    constexpr int kWarps = NT / 32;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float w = __shfl_xor_sync(0xffffffffu, v, o);
        v = MAX ? fmaxf(v, w) : v + w;
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) r = MAX ? fmaxf(r, red[w]) : r + red[w];
    __syncthreads();  // red[] is reused by the next reduction
    return r;
}

template <int D, int NT>
__global__ void __launch_bounds__(NT, 512 / NT) q4_flash_combine_kernel(const __grid_constant__ FdParams p) {
    // Chunk c belongs to class c % kRes; every class is summed in increasing chunk order into its
    // own accumulator and the classes are added in class order -- the same sums, in the same
    // order, for either thread count, so the result does not depend on NT.
    constexpr int kRes = 512 / D;        // classes
    constexpr int kSplit = NT / D;       // threads per output element
    constexpr int kMine = kRes / kSplit; // classes per thread: j, j + kSplit, ...
    constexpr int kAhead = 48 / kMine;   // partials per class per round, all loaded before any use
    constexpr int kPer = kFdMaxChunks / NT;
    __shared__ float w_s[kFdMaxChunks];  // chunk maxima, then weights 2^(m_c - M)
    __shared__ float l_s[kFdMaxChunks];  // chunk sums l_c
    __shared__ float red[NT / 32];
    __shared__ float osum[kRes][D];
    __shared__ float lsum[kRes];
    grid_dependency_wait();  // the chunk partials
    allow_dependents();
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const int g = p.g, kvh = h / g, row = h - kvh * g;
    const size_t slot0 = (static_cast<size_t>(b) * p.Hkv + kvh) * p.C * g + row;  // chunk c: + c*g
    const int j = tid / D, e = tid - j * D;

    // a round: entry e of chunks cls + (r0 + i) kRes of this thread's classes, below `bound`
    float v[kMine][kAhead];
    auto load_round = [&](int r0, int bound) {
#pragma unroll
        for (int k = 0; k < kMine; ++k)
#pragma unroll
            for (int i = 0; i < kAhead; ++i) {
                const int c = j + k * kSplit + (r0 + i) * kRes;
                v[k][i] = c < bound ? ld_dep_f32(p.part + (slot0 + static_cast<size_t>(c) * g) * D + e) : 0.f;
            }
    };
    // The first round of partials and every chunk's (m, l) are loaded together with the length
    // (one memory round trip, not two), bounded by the chunk capacity C: entries of chunks at or
    // past the used count hold stale workspace data and are never read back below.
    int len, cs, used;
    fd_chunking(p, b, len, cs, used);
    load_round(0, p.C);
    float mraw[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int c = tid + i * NT;
        mraw[i] = -INFINITY;
        if (c < p.C) {
            const uint2 ml = ld_dep_u2(p.ml + (slot0 + static_cast<size_t>(c) * g) * 2);
            mraw[i] = __uint_as_float(ml.x);
            l_s[c] = __uint_as_float(ml.y);
        }
    }
    float* out = p.O + (static_cast<size_t>(b) * p.Hkv * g + h) * D;
    if (used == 0) {  // empty cache: O = 0
        if (tid < D) out[tid] = 0.f;
        return;
    }
    float mmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int c = tid + i * NT;
        if (c < used) {
            w_s[c] = mraw[i];
            mmax = fmaxf(mmax, mraw[i]);
        }
    }
    const float M = block_reduce<true, NT>(mmax, red);  // a maximum: exact in any order
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int c = tid + i * NT;
        if (c < used) w_s[c] = ex2(w_s[c] - M);
    }
    __syncthreads();

    float o[kMine], l[kMine];
#pragma unroll
    for (int k = 0; k < kMine; ++k) o[k] = l[k] = 0.f;
    for (int r0 = 0;;) {
#pragma unroll
        for (int k = 0; k < kMine; ++k)
#pragma unroll
            for (int i = 0; i < kAhead; ++i) {
                const int c = j + k * kSplit + (r0 + i) * kRes;
                if (c < used) {
                    o[k] = fmaf(w_s[c], v[k][i], o[k]);
                    l[k] = fmaf(w_s[c], l_s[c], l[k]);
                }
            }
        r0 += kAhead;
        if (r0 * kRes >= used) break;
        load_round(r0, used);
    }
#pragma unroll
    for (int k = 0; k < kMine; ++k) {
        osum[j + k * kSplit][e] = o[k];
        if (e == 0) lsum[j + k * kSplit] = l[k];
    }
    __syncthreads();
    if (tid < D) {
        float r = osum[0][tid], L = lsum[0];
#pragma unroll
        for (int i = 1; i < kRes; ++i) {
            r += osum[i][tid];
            L += lsum[i];
        }
        out[fd_dim(tid)] = r / L;
    }
}

// raise a kernel's dynamic shared memory limit once per (kernel, device) when it needs more than
// the default 48 KB
bool smem_limit_raised(void (*fn)(FdParams), size_t bytes) {
    if (bytes <= 48 * 1024) return true;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    static std::mutex mu;
    static std::set<std::pair<const void*, int>> done;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_pair(reinterpret_cast<const void*>(fn), dev);
    if (done.count(key)) return true;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) !=
        cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    done.insert(key);
    return true;
}

bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// CTAs of the split kernel resident per SM with this much dynamic shared memory (cached per
// kernel, size and device; 0 on error)
int resident_ctas(void (*fn)(FdParams), size_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    static std::mutex mu;
    static std::map<std::tuple<const void*, size_t, int>, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_tuple(reinterpret_cast<const void*>(fn), smem, dev);
    const auto hit = cache.find(key);
    if (hit != cache.end()) return hit->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kFdWarps * 32, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cache[key] = n;
    return n;
}

// how the split kernel fills its ring: one bulk copy per row (default) or per-lane 16-byte
// cp.async (Q4_FD_BULK=0); both give the same bits
bool fd_bulk() {
    const char* v = std::getenv("Q4_FD_BULK");
    return !(v && *v && std::atoi(v) == 0);
}

// threads per combine CTA for this many (query head, sequence) pairs (Q4_FD_COMBINE = 256 or
// 512 overrides)
int fd_combine_threads(int64_t pairs, int sms) {
    const char* v = std::getenv("Q4_FD_COMBINE");
    if (v && *v) return std::atoi(v) == 256 ? 256 : 512;
    return pairs <= sms ? 512 : 256;
}

// ring slots per warp of the cp.async fill (Q4_FD_STAGES = 2 or 3)
int fd_stages() {
    const char* v = std::getenv("Q4_FD_STAGES");
    return v && std::atoi(v) == 2 ? 2 : kFdStages;
}

int fd_chunks(int n_kv_heads, int n_chunks, int sms) {
    if (n_chunks > 0) return n_chunks;
    // about eight chunks per SM for one sequence (chunks are still at least kFdMinChunk long)
    const int c = (8 * sms) / n_kv_heads;
    return c < 1 ? 1 : (c > kFdMaxChunks ? kFdMaxChunks : c);
}

size_t fd_part_bytes(int B, int Hq, int D, int C) {
    const size_t v = static_cast<size_t>(B) * Hq * C * D * sizeof(float);
    return (v + 255) / 256 * 256;
}

q4_status fd_check(int B, int Hq, int Hkv, int D, int n_chunks) {
    if (B < 1 || B > 65535 || Hkv < 1 || Hkv > 65535 || Hq < 1 || Hq % Hkv != 0 || Hq / Hkv > kFdMaxGroup ||
        n_chunks < 0 || n_chunks > kFdMaxChunks)
        return Q4_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return Q4_ERR_UNSUPPORTED_SHAPE;
    return Q4_OK;
}

}  // namespace

int q4i_attn_take_error() {
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_fd_device_error, sizeof v) != cudaSuccess) return -1;
    if (v == 0) return 0;
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_fd_device_error, &zero, sizeof zero) != cudaSuccess) return -1;
    return 1;
}

// ------------------------------------------------------------------ C ABI
extern "C" int q4_flash_decode_chunks(int n_kv_heads, int n_chunks) {
    if (n_kv_heads < 1 || n_chunks < 0 || n_chunks > kFdMaxChunks) return 0;
    if (n_chunks > 0) return n_chunks;
    const int sms = q4i_sm_count(nullptr);
    return sms > 0 ? fd_chunks(n_kv_heads, 0, sms) : 0;
}

extern "C" size_t q4_flash_decode_workspace_bytes(int B, int n_q_heads, int n_kv_heads, int head_dim,
                                                  int n_chunks) {
    if (fd_check(B, n_q_heads, n_kv_heads, head_dim, n_chunks) != Q4_OK) return 0;
    const int C = q4_flash_decode_chunks(n_kv_heads, n_chunks);
    if (C <= 0) return 0;
    return fd_part_bytes(B, n_q_heads, head_dim, C) + static_cast<size_t>(B) * n_q_heads * C * 2 * sizeof(float);
}

extern "C" q4_status q4_flash_decode(const uint16_t* Q, const uint16_t* K_cache, const uint16_t* V_cache,
                                     const int32_t* lengths, int B, int n_q_heads, int n_kv_heads, int head_dim,
                                     int64_t max_len, float scale, int n_chunks, float* O, void* ws,
                                     size_t ws_bytes, void* stream) {
    if (!Q || !K_cache || !V_cache || !lengths || !O || !ws) return Q4_ERR_INVALID_ARG;
    const q4_status st = fd_check(B, n_q_heads, n_kv_heads, head_dim, n_chunks);
    if (st != Q4_OK) return st;
    if (max_len < 1 || max_len > kFdMaxLen || !std::isfinite(scale)) return Q4_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(K_cache, 16) || !aligned(V_cache, 16) || !aligned(ws, 16) ||
        !aligned(O, 4) || !aligned(lengths, 4))
        return Q4_ERR_MISALIGNED;
    int sms = 0;
    int C = n_chunks;
    if (C == 0) {  // the default count needs the device's SM count
        sms = q4i_sm_count(nullptr);
        if (sms <= 0) return Q4_ERR_CUDA;
        C = fd_chunks(n_kv_heads, 0, sms);
        // no more chunks than a max_len cache has at the minimum length: every chunk stays
        // kFdMinChunk long either way (ceil(len / C) <= kFdMinChunk for len <= max_len), so the
        // result is the same, and the combine looks at fewer chunk slots
        const int64_t short_c = (max_len + kFdMinChunk - 1) / kFdMinChunk;
        if (short_c < C) C = static_cast<int>(short_c);
    }
    const size_t need = fd_part_bytes(B, n_q_heads, head_dim, C) +
                        static_cast<size_t>(B) * n_q_heads * C * 2 * sizeof(float);
    if (ws_bytes < need) return Q4_ERR_WORKSPACE;
    if (q4i_fault_injected()) return Q4_ERR_CUDA;
    if (sms == 0) {
        sms = q4i_sm_count(nullptr);
        if (sms <= 0) return Q4_ERR_CUDA;
    }

    FdParams p{};
    p.Q = Q;
    p.K = K_cache;
    p.V = V_cache;
    p.lengths = lengths;
    p.O = O;
    p.part = static_cast<float*>(ws);
    p.ml = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + fd_part_bytes(B, n_q_heads, head_dim, C));
    p.Lmax = max_len;
    p.c = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);  // scale * log2(e)
    p.Hkv = n_kv_heads;
    p.g = n_q_heads / n_kv_heads;
    p.C = C;
    p.min_chunk = kFdMinChunk;


    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 1;

    cfg.gridDim = dim3(1u, static_cast<unsigned>(n_kv_heads), static_cast<unsigned>(B));
    cfg.blockDim = dim3(kFdWarps * 32);
    const bool bulk = fd_bulk();
    const int stages = bulk ? kFdStages : fd_stages();
    const int slot = head_dim == 64 ? (bulk ? FdSlot<64, true>::kBytes : FdSlot<64, false>::kBytes)
                                    : (bulk ? FdSlot<128, true>::kBytes : FdSlot<128, false>::kBytes);
    cfg.dynamicSmemBytes = static_cast<size_t>(kFdWarps) * stages * (slot + (bulk ? 8 : 0));
    using SplitFn = void (*)(FdParams);
    const SplitFn split =
        head_dim == 64 ? (bulk ? q4_flash_split_kernel<64, kFdStages, true>
                               : stages == 2 ? q4_flash_split_kernel<64, 2, false> : q4_flash_split_kernel<64, 3, false>)
                       : (bulk ? q4_flash_split_kernel<128, kFdStages, true>
                               : stages == 2 ? q4_flash_split_kernel<128, 2, false>
                                             : q4_flash_split_kernel<128, 3, false>);
    if (!smem_limit_raised(split, cfg.dynamicSmemBytes)) return Q4_ERR_CUDA;
    // CTAs per (sequence, KV head): enough warps for the most chunks any sequence can have, and
    // one full wave of resident CTAs over the batch (this choice changes no result)
    const int resident = resident_ctas(split, cfg.dynamicSmemBytes);
    if (resident <= 0) return Q4_ERR_CUDA;
    const int64_t most = std::min<int64_t>(C, (max_len + kFdMinChunk - 1) / kFdMinChunk);
    const int64_t fill = std::max<int64_t>(1, (static_cast<int64_t>(resident) * sms) / (static_cast<int64_t>(B) * n_kv_heads));
    const int64_t per_head = std::max<int64_t>(1, std::min<int64_t>(fill, (most + kFdWarps - 1) / kFdWarps));
    cfg.gridDim.x = static_cast<unsigned>(per_head);
    if (cudaLaunchKernelEx(&cfg, split, p) != cudaSuccess) return Q4_ERR_CUDA;

    // combine: 512-thread CTAs (one per SM) while the (query head, sequence) pairs fit in one
    // wave, else 256-thread CTAs (two per SM); the order of every sum is fixed by D and the
    // thread count, and so by B and the SM count only
    const int nt = fd_combine_threads(static_cast<int64_t>(B) * n_q_heads, sms);
    cfg.gridDim = dim3(static_cast<unsigned>(n_q_heads), static_cast<unsigned>(B));
    cfg.blockDim = dim3(static_cast<unsigned>(nt));
    cfg.dynamicSmemBytes = 0;
    using CombineFn = void (*)(FdParams);
    const CombineFn comb = head_dim == 64 ? (nt == 512 ? q4_flash_combine_kernel<64, 512> : q4_flash_combine_kernel<64, 256>)
                                          : (nt == 512 ? q4_flash_combine_kernel<128, 512>
                                                       : q4_flash_combine_kernel<128, 256>);
    return cudaLaunchKernelEx(&cfg, comb, p) == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}
