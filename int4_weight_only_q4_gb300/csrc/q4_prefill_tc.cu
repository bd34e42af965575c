// int4 prefill GEMM on the fifth-generation tensor cores of sm_103a: tcgen05.mma with its
// accumulators in tensor memory (TMEM), activations brought in by TMA.
//
// What is computed (the rumik-oss-1 int4 engine write-up, rtts.neoandmatrix.me, "Step 8: a
// prefill that stays int4": the weights stay 4-bit, each group is expanded for the tensor cores
// and its scale and minimum are applied to the fp32 result):
//     Y[m, n] = sum_g ( scale[n, g] * sum_{k in g} code[n, k] x[m, k]  +  min[n, g] * sum_{k in g} x[m, k] )
// for a prompt of M tokens, g = k / 128, fp32 accumulation.
//
// Operands.  A code becomes an exact bf16 operand with one AND per two codes, as in the GEMV
// kernels: a bf16 whose exponent field is 0 or 1 and whose low 8 bits hold m is exactly
// m * 2^-133, so for a 32-bit word w of packed codes (bytes b0..b3, low nibble first)
//     w & 0x000F000F          holds (code k+0, code k+4)
//     w & 0x00F000F0          holds (code k+1, code k+5) times 16
//     (w >> 8) & 0x000F000F   holds (code k+2, code k+6)
//     (w >> 8) & 0x00F000F0   holds (code k+3, code k+7) times 16
// and these four registers, stored in that order, are four consecutive TMEM columns of one A row
// (two bf16 per column) whose 8 slots hold the codes of k + [0, 4, 1, 5, 2, 6, 3, 7].  The activations are stored with the same
// slot order (a dot product does not depend on the order of k as long as both operands share it),
// scaled per token by 2^a (slots of even k) or 2^(a-4) (slots of odd k, where the codes carry the
// factor 16), so that every product is a normal fp32 number; q4_tc_prep_kernel writes that copy
// X' of the tokens, the group sums S' = S * 2^(a-133) and the token factors f = 2^(133-a).
// Every step is exact but the fp32 sums; the result is f * sum_g (scale D_g + min S'_g).
//
// The CTA computes a 128-row x 128-token tile of Y (grid: row blocks fastest, then token tiles).
// The expanded codes (the A operand) live in TMEM, not in shared memory: an MMA of 128 x 128 x 16
// that read both operands from shared memory would by itself use all of an SM's shared-memory
// bandwidth, leaving none for the copies that feed it.  Warp roles (14 warps):
//   warp 0       TMA: per half-group (64 k) the 128-token x 64 activation box (SWIZZLE_128B) into a
//                shared-memory ring of kBStages slots, and per group the tile's 128 group sums into
//                a ring of kSumSlots slots that the epilogue frees;
//   warp 1       allocates all 512 TMEM columns; one thread issues, per group, 8 tcgen05.mma
//                (128 x 128 x 16, A from TMEM, B from shared memory) into accumulator buffer g % kDBufs,
//                frees the A and B stages with tcgen05.commit, and signals the epilogue with another;
//                it reads no memory between MMAs (a load would stall it until its MMAs drain) and
//                learns that a group may go from a named barrier;
//   warp 14      scheduler: waits on the mbarriers that gate a step and releases it to warp 1;
//   warps 2..5   code expansion: thread = weight row 32 (w % 4) + lane; per group its 64 code bytes
//                (loaded three groups ahead) become 64 TMEM columns (tcgen05.st) in a ring of
//                kAStages half-group stages of 32 columns;
//   warps 6..13  the epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 (weight rows) and 64
//                token columns (4 x tcgen05.ld 32x32b.x16), releases the buffer, then
//                acc = fma(scale, D, acc); acc = fma(min, S', acc) for its row and 64 tokens; at
//                the end y = acc * f.
// Every wait is bounded; one that gives up sets a device error word (read by q4_device_status)
// and a CTA-wide abort flag that makes every other wait of the CTA return, so the CTA still frees
// its TMEM and exits.
#include <cuda.h>  // CUtensorMap and its enums; the encoder is looked up through the runtime
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "q4.h"
#include "q4_common.cuh"

namespace {

constexpr int kTcRows = 128;                   // weight rows per CTA (MMA M)
constexpr int kTcTok = 128;                    // tokens per CTA (MMA N)
constexpr int kBStages = 8;                    // shared-memory ring of activation boxes, one half-group (64 k) each
constexpr int kAStages = 4;                    // TMEM ring of expanded codes, one half-group each (32 columns)
constexpr int kDBufs = 3;                      // TMEM accumulator buffers (128 columns each)
constexpr int kSlotBytes = 128 * 64 * 2;       // 128 tokens x 64 bf16: 16 KB
constexpr int kSumSlots = 8;                   // ring of group sums (128 floats each) for the epilogue
constexpr int kTcRecBytes = 1088;              // one tiled record (16 rows x 128 columns + scale/min)
constexpr int kTcThreads = 480;                // 15 warps
constexpr int kStepBar = 1;                    // named barrier: scheduler and MMA warps meet once per step
constexpr int kTmemCols = 512;                 // kDBufs x 128 accumulator columns + kAStages x 32 A columns
constexpr uint32_t kTcWaitLimit = 1u << 22;
constexpr size_t kTcSmem = kBStages * kSlotBytes + kSumSlots * 512 + 512 + 1024;  // + barriers, TMEM address, alignment
static_assert(kDBufs * kTcTok + kAStages * 32 <= kTmemCols, "TMEM budget");

__device__ unsigned int g_tc_device_error;

struct TcParams {
    const uint8_t* tiled;  // tiled copy of the weights
    const float* ssum;     // [token tiles][G][128]: group sums times 2^(a-133)
    const float* fac;      // [token tiles * 128]: 2^(133-a) per token
    float* y;              // [M, N]
    int N, K, M;
    int row_blocks;
};

// ---- tcgen05 / TMA primitives (inline PTX)
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row groups 1,024 bytes
// apart (stride byte offset), leading byte offset unused for this layout (encoded as 1), version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both K-major, N and M.
__host__ __device__ constexpr uint32_t tc_idesc(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

// Arrive on `bar` once every tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&d)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]), "=r"(d[4]), "=r"(d[5]), "=r"(d[6]), "=r"(d[7]),
          "=r"(d[8]), "=r"(d[9]), "=r"(d[10]), "=r"(d[11]), "=r"(d[12]), "=r"(d[13]), "=r"(d[14]), "=r"(d[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 2-D TMA load of one box into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ uint32_t ld_nc_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
// Read-only 16-byte load that may stay in L1 (a row's four pieces share cache lines with its
// neighbours' pieces).
__device__ __forceinline__ uint4 ld_nc_u4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ float half_lo(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
}

// A bounded wait that gives up at once when the CTA has aborted, and aborts the CTA when it runs
// out (the error word tells the host).
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    const uint32_t a = smem_addr(bar);
    for (uint32_t it = 0; it < kTcWaitLimit; ++it) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
        if ((it & 255u) == 255u && *abort_flag) return false;
    }
    *abort_flag = 1;
    atomicOr(&g_tc_device_error, 1u);
    return false;
}

// The same wait taken by a whole converged warp: every lane gets the same answer.
__device__ __forceinline__ bool tc_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    return __all_sync(0xffffffffu, tc_wait(bar, parity, abort_flag));
}

// A 128 x 64 (k) activation slot with 128-byte swizzle, as TMA writes it: row r, 16-byte chunk c
// (0..7) at (r / 8) * 1024 + (r % 8) * 128 + ((c ^ (r % 8)) * 16).  The descriptor above describes it.

// Store 16 consecutive 32-bit TMEM columns of this thread's lane (warp w reaches lanes 32 (w % 4) ..).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// A operand in TMEM: D += A B with A (128 x 16, one row per lane, 8 columns of bf16 pairs) at a_tmem.
__device__ __forceinline__ void tc_mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                          uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// Codes of one row, 32 of them in a 16-byte piece (4 words of 8), as 16 TMEM columns: word i gives
// the columns 4i .. 4i+3 (slots k+0,k+4 | k+1,k+5 | k+2,k+6 | k+3,k+7, see the file comment).
__device__ __forceinline__ void expand32(const uint4& v, uint32_t (&o)[16]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w8 = w[i] >> 8;
        o[4 * i + 0] = w[i] & 0x000F000Fu;
        o[4 * i + 1] = w[i] & 0x00F000F0u;
        o[4 * i + 2] = w8 & 0x000F000Fu;
        o[4 * i + 3] = w8 & 0x00F000F0u;
    }
}

__global__ void __launch_bounds__(kTcThreads, 1) q4_prefill_tc_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                      const __grid_constant__ TcParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    unsigned char* sB = smem;                                     // kBStages x 16 KB
    float* sS = reinterpret_cast<float*>(smem + kBStages * kSlotBytes);  // kSumSlots x 128 sums
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<unsigned char*>(sS) + kSumSlots * 512);
    uint64_t* fullA = bars;                      // unpack warps (4) -> MMA, per TMEM A stage
    uint64_t* emptyA = fullA + kAStages;         // MMA commit -> unpack warps
    uint64_t* fullB = emptyA + kAStages;         // TMA bytes -> MMA, per smem B stage
    uint64_t* emptyB = fullB + kBStages;         // MMA commit -> TMA
    uint64_t* dfull = emptyB + kBStages;         // MMA commit -> epilogue, per accumulator buffer
    uint64_t* dempty = dfull + kDBufs;           // epilogue (8 warps) -> MMA
    uint64_t* sfull = dempty + kDBufs;           // group sums landed, per sum slot
    uint64_t* sempty = sfull + kSumSlots;        // epilogue (8 warps) done with a sum slot
    uint64_t* fin = sempty + kSumSlots;          // all MMAs done (teardown)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = static_cast<int>(threadIdx.x) >> 5, lane = static_cast<int>(threadIdx.x) & 31;
    const int G = p.K >> 7, H = 2 * G;
    const int rb = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.row_blocks));
    const int tt = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.row_blocks));
    const int row0 = rb * kTcRows, tok0 = tt * kTcTok;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kAStages; ++s) {
            mbar_init(fullA + s, 4);
            mbar_init(emptyA + s, 1);
        }
        for (int s = 0; s < kBStages; ++s) {
            mbar_init(fullB + s, 1);
            mbar_init(emptyB + s, 1);
        }
        for (int b = 0; b < kDBufs; ++b) {
            mbar_init(dfull + b, 1);
            mbar_init(dempty + b, 8);
        }
        for (int e = 0; e < kSumSlots; ++e) {
            mbar_init(sfull + e, 1);
            mbar_init(sempty + e, 8);
        }
        mbar_init(fin, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmemA = tmem + kDBufs * kTcTok;  // A stages: 32 columns each

    if (warp == 0) {
        // ---- TMA producer (one thread): per half-group the activation box, per group its sums
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
            grid_dependency_wait();  // X', the sums and the factors come from the prep kernel
            const float* sums = p.ssum + static_cast<size_t>(tt) * G * kTcTok;
            int issued = 0, sums_issued = 0;
            for (int h = 0; h < H; ++h) {
                const int s = h % kBStages;
                if (!tc_wait(emptyB + s, (static_cast<uint32_t>(h / kBStages) & 1u) ^ 1u, abort_flag)) break;
                mbar_arrive_expect_tx(fullB + s, kSlotBytes);
                tma_load_2d(sB + s * kSlotBytes, &xmap, 64 * h, tok0, fullB + s);
                issued = h + 1;
                if ((h & 1) == 0) {
                    const int g = h >> 1, e = g % kSumSlots;
                    if (!tc_wait(sempty + e, (static_cast<uint32_t>(g / kSumSlots) & 1u) ^ 1u, abort_flag)) break;
                    mbar_arrive_expect_tx(sfull + e, 512u);
                    bulk_g2s(sS + e * kTcTok, sums + static_cast<size_t>(g) * kTcTok, 512u, sfull + e);
                    sums_issued = g + 1;
                }
            }
            // copies still in flight land before the CTA leaves (at once on the normal path)
            for (int h = issued - kBStages < 0 ? 0 : issued - kBStages; h < issued; ++h)
                (void)mbar_wait(fullB + h % kBStages, static_cast<uint32_t>(h / kBStages) & 1u, kTcWaitLimit);
            for (int g = sums_issued - kSumSlots < 0 ? 0 : sums_issued - kSumSlots; g < sums_issued; ++g)
                (void)mbar_wait(sfull + g % kSumSlots, static_cast<uint32_t>(g / kSumSlots) & 1u, kTcWaitLimit);
        }
    } else if (warp == 1) {
        // ---- MMA issue (one thread).  This warp reads no memory while its MMAs run: a load (shared or
        // global, by any lane, an mbarrier wait included) stalls the warp until its MMAs in flight have
        // drained, about 380 cycles each time.  The scheduler warp (14) does the waiting; the two warps
        // meet at named barrier kStepBar once per group (a strict rendezvous, so no step is skipped or
        // taken twice), and the scheduler meets it at every step, also after a wait gave up, so this
        // warp never blocks for good.
        constexpr uint32_t idesc = tc_idesc(kTcRows, kTcTok);
        const uint64_t bd0 = sw128_desc(smem_addr(sB));
        for (int g = 0; g < G; ++g) {  // one step per group: its two half-groups, 8 MMAs
            asm volatile("bar.sync %0, 64;" ::"n"(kStepBar) : "memory");
            tc_fence_after();
            if (lane == 0) {
                const uint32_t d = tmem + static_cast<uint32_t>((g % kDBufs) * kTcTok);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int h = 2 * g + hf, sa = h % kAStages, sb = h % kBStages;
                    const uint64_t bd = bd0 + static_cast<uint64_t>((sb * kSlotBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)  // K = 16 per instruction: 8 A columns, 32 bytes of each B row
                        tc_mma_ta(d, tmemA + static_cast<uint32_t>(32 * sa + 8 * kk), bd + static_cast<uint64_t>(2 * kk),
                                  idesc, (hf | kk) != 0 ? 1u : 0u);
                    tc_commit(emptyA + sa);  // the stages are free once these MMAs have read them
                    tc_commit(emptyB + sb);
                }
                tc_commit(dfull + g % kDBufs);
            }
            __syncwarp();
        }
        // every MMA this thread issued has completed before TMEM is freed (at once on the normal path)
        if (lane == 0) {
            tc_commit(fin);
            (void)mbar_wait(fin, 0u, kTcWaitLimit);
        }
        __syncwarp();
    } else if (warp == 14) {
        // ---- scheduler: per group, the accumulator buffer is free, both half-groups' codes are in TMEM
        // and their activations have landed; then the MMA warp may issue the group
        // The five waits of a step run side by side, one lane each (lane 0: the accumulator buffer;
        // lanes 1-4: codes and activations of the two half-groups): a wait costs a few hundred cycles
        // even on a completed phase, so five in sequence were most of a step's time.  The warp
        // barrier after them orders every lane's acquire before the named barrier that releases
        // the MMA warp.
        bool aborted = false;
        for (int g = 0; g < G; ++g) {
            if (!aborted) {  // after a wait gave up, the remaining steps go on garbage (the error word is set)
                bool ok = true;
                if (lane < 5) {
                    uint64_t* bar;
                    uint32_t parity;
                    if (lane == 0) {
                        bar = dempty + g % kDBufs;
                        parity = (static_cast<uint32_t>(g / kDBufs) & 1u) ^ 1u;
                    } else {
                        const int h = 2 * g + ((lane - 1) >> 1);
                        if (((lane - 1) & 1) == 0) {
                            bar = fullA + h % kAStages;
                            parity = static_cast<uint32_t>(h / kAStages) & 1u;
                        } else {
                            bar = fullB + h % kBStages;
                            parity = static_cast<uint32_t>(h / kBStages) & 1u;
                        }
                    }
                    ok = tc_wait(bar, parity, abort_flag);
                }
                __syncwarp();
                aborted = !__all_sync(0xffffffffu, ok);
            }
            asm volatile("bar.sync %0, 64;" ::"n"(kStepBar) : "memory");
        }
    } else if (warp < 6) {
        // ---- code expansion into TMEM: thread = weight row 32 (warp % 4) + lane of the CTA's 128; per
        // group its 64 code bytes (one 16-row record holds row q's at 64 q, row q+8's at 512 + 64 q),
        // loaded three groups ahead, become 64 TMEM columns of bf16 pairs (two half-group stages)
        const int r = 32 * (warp & 3) + lane, n = row0 + r;
        const bool row_ok = n < p.N;
        const int rr = n & 15;
        const uint8_t* src = p.tiled + static_cast<size_t>(row_ok ? (n >> 4) : 0) * G * kTcRecBytes +
                             (rr < 8 ? 64 * rr : 512 + 64 * (rr - 8));
        const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        uint4 cur[4], nx1[4], nx2[4];
        auto load = [&](int g, uint4 (&v)[4]) {  // weights are read-only: no wait for the kernel before
#pragma unroll
            for (int c = 0; c < 4; ++c)
                v[c] = (row_ok && g < G) ? ld_nc_u4(src + static_cast<size_t>(g) * kTcRecBytes + 16 * c)
                                         : make_uint4(0u, 0u, 0u, 0u);
        };
        load(0, cur);
        load(1, nx1);
        load(2, nx2);
        for (int g = 0; g < G; ++g) {
            uint4 nn[4];
            load(g + 3, nn);
            bool ok = true;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int h = 2 * g + hf, sa = h % kAStages;
                ok = ok && tc_wait_warp(emptyA + sa, (static_cast<uint32_t>(h / kAStages) & 1u) ^ 1u, abort_flag);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {  // the half-group's 64 codes: two 16-byte pieces
                    uint32_t o[16];
                    expand32(cur[2 * hf + c2], o);
                    tmem_st16(tmemA + lane_off + static_cast<uint32_t>(32 * sa + 16 * c2), o);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(fullA + sa);
            }
            if (!ok) break;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                cur[c] = nx1[c];
                nx1[c] = nx2[c];
                nx2[c] = nn[c];
            }
        }
    } else {
        // ---- epilogue: TMEM lanes 32 (warp % 4) .. + 31, token columns 64 ch .. + 63
        grid_dependency_wait();  // Y may still be read or written by the kernel before; f comes from the prep
        const int lq = warp & 3, ch = (warp - 6) >> 2;
        const int r = 32 * lq + lane, n = row0 + r;
        const bool row_ok = n < p.N;
        const int tile = n >> 4, rr = n & 15;
        // scale | min << 16 of row n in record (tile, g), loaded three groups ahead
        const uint8_t* smw_ptr =
            p.tiled + static_cast<size_t>(row_ok ? tile : 0) * G * kTcRecBytes + 1024 + 8 * (rr & 7) + 4 * (rr >> 3);
        auto smw_load = [&](int g) -> uint32_t {
            return (row_ok && g < G) ? ld_nc_u32(smw_ptr + static_cast<size_t>(g) * kTcRecBytes) : 0u;
        };
        uint32_t sq0 = smw_load(0), sq1 = smw_load(1), sq2 = smw_load(2);
        float acc[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) acc[j] = 0.f;
        bool ok = true;
        for (int g = 0; g < G && ok; ++g) {
            const int b = g % kDBufs, e = g % kSumSlots;
            const uint32_t smw = sq0;
            sq0 = sq1;
            sq1 = sq2;
            sq2 = smw_load(g + 3);
            ok = tc_wait_warp(dfull + b, static_cast<uint32_t>(g / kDBufs) & 1u, abort_flag) &&
                 tc_wait_warp(sfull + e, static_cast<uint32_t>(g / kSumSlots) & 1u, abort_flag);
            if (!ok) break;
            tc_fence_after();
            uint32_t d[4][16];
            const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * lq) << 16) + static_cast<uint32_t>(b * kTcTok + 64 * ch);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) tmem_ld16(taddr + 16 * c4, d[c4]);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dempty + b);  // the buffer may take group g + kDBufs
            const float sc = half_lo(smw), mn = half_lo(smw >> 16);
            const float* Sg = sS + e * kTcTok + 64 * ch;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
#pragma unroll
                for (int j = 0; j < 16; j += 4) {
                    const float4 s4 = *reinterpret_cast<const float4*>(Sg + 16 * c4 + j);
                    const int o = 16 * c4 + j;
                    acc[o + 0] = fmaf(sc, __uint_as_float(d[c4][j + 0]), acc[o + 0]);
                    acc[o + 0] = fmaf(mn, s4.x, acc[o + 0]);
                    acc[o + 1] = fmaf(sc, __uint_as_float(d[c4][j + 1]), acc[o + 1]);
                    acc[o + 1] = fmaf(mn, s4.y, acc[o + 1]);
                    acc[o + 2] = fmaf(sc, __uint_as_float(d[c4][j + 2]), acc[o + 2]);
                    acc[o + 2] = fmaf(mn, s4.z, acc[o + 2]);
                    acc[o + 3] = fmaf(sc, __uint_as_float(d[c4][j + 3]), acc[o + 3]);
                    acc[o + 3] = fmaf(mn, s4.w, acc[o + 3]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sempty + e);  // the sum slot may take group g + kSumSlots
        }
        if (ok && row_ok) {
            const int m0 = tok0 + 64 * ch;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const int m = m0 + j;
                if (m < p.M) p.y[static_cast<size_t>(m) * p.N + n] = acc[j] * ld_dep_f32(p.fac + m);
            }
        }
    }
    allow_dependents();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// ---- activation prep: one CTA of 128 threads per token (rows M .. M_pad-1 write zero sums and
// factors).  a = clamp(120 - e, 6, 253), e = the exponent of the row's largest |x| (the rule of the
// GEMV kernels); X'[m, 8j + s] = x[m, 8j + pi(s)] * (pi(s) even ? 2^a : 2^(a-4)), pi = 0 4 1 5 2 6 3 7;
// S'[m, g] = (sum of the group's 128 x in a fixed order) * 2^(a-133); f[m] = 2^(133-a).
__global__ void __launch_bounds__(128) q4_tc_prep_kernel(const uint16_t* __restrict__ x, int K, int M,
                                                         uint16_t* __restrict__ xp, float* __restrict__ ssum,
                                                         float* __restrict__ fac) {
    __shared__ unsigned red[4];
    grid_dependency_wait();  // x may be the previous kernel's output; the outputs may still be read
    allow_dependents();
    const int m = static_cast<int>(blockIdx.x), tid = static_cast<int>(threadIdx.x);
    const int G = K >> 7, tt = m / kTcTok, mr = m % kTcTok;
    if (m >= M) {
        for (int g = tid; g < G; g += 128) ssum[(static_cast<size_t>(tt) * G + g) * kTcTok + mr] = 0.f;
        if (tid == 0) fac[m] = 0.f;
        return;
    }
    const uint4* row = reinterpret_cast<const uint4*>(x + static_cast<size_t>(m) * K);
    const int chunks = K >> 3;  // 16-byte pieces of 8 values
    unsigned mx = 0;
    for (int c = tid; c < chunks; c += 128) {
        const uint4 v = row[c];
        const uint32_t h[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) mx = max(mx, max((h[e] << 16) & 0x7FFFFFFFu, h[e] & 0x7FFF0000u));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((tid & 31) == 0) red[tid >> 5] = mx;
    __syncthreads();
    mx = max(max(red[0], red[1]), max(red[2], red[3]));
    const int e = static_cast<int>(mx >> 23) - 127;  // mx == 0: e = -127
    int a = 120 - e;
    a = a < 6 ? 6 : (a > 253 ? 253 : a);
    const int a1 = a > 127 ? 127 : a;
    const float m1 = __int_as_float((a1 + 127) << 23), m2 = __int_as_float((a - a1 + 127) << 23);
    uint4* out = reinterpret_cast<uint4*>(xp + static_cast<size_t>(m) * K);
    // warp w takes groups w, w + 4, ...; lanes 0-15 one group's 16 pieces, lanes 16-31 the next's
    const int w = tid >> 5, l = tid & 31;
    for (int g0 = 2 * w; g0 < G; g0 += 8) {
        const int g = g0 + (l >> 4);
        float s = 0.f;
        if (g < G) {
            const int c = g * 16 + (l & 15);
            const uint4 v = row[c];
            s = __uint_as_float(v.x << 16);
            s += __uint_as_float(v.x & 0xFFFF0000u);
            s += __uint_as_float(v.y << 16);
            s += __uint_as_float(v.y & 0xFFFF0000u);
            s += __uint_as_float(v.z << 16);
            s += __uint_as_float(v.z & 0xFFFF0000u);
            s += __uint_as_float(v.w << 16);
            s += __uint_as_float(v.w & 0xFFFF0000u);
            // slots: (k0, k4) (k1, k5) (k2, k6) (k3, k7); odd k carry 2^(a-4)
            const uint32_t p0 = bf16x2_scale(__byte_perm(v.x, v.z, 0x5410), m1, m2);
            const uint32_t p1 = bf16x2_scale(__byte_perm(v.x, v.z, 0x7632), m1, m2 * 0.0625f);
            const uint32_t p2 = bf16x2_scale(__byte_perm(v.y, v.w, 0x5410), m1, m2);
            const uint32_t p3 = bf16x2_scale(__byte_perm(v.y, v.w, 0x7632), m1, m2 * 0.0625f);
            out[c] = make_uint4(p0, p1, p2, p3);
        }
        s += __shfl_xor_sync(0xffffffffu, s, 8);
        s += __shfl_xor_sync(0xffffffffu, s, 4);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        if (g < G && (l & 15) == 0) {
            const int ee = a - 133, e1 = ee < -63 ? -63 : ee, e2 = ee - e1;
            ssum[(static_cast<size_t>(tt) * G + g) * kTcTok + mr] =
                (s * __int_as_float((e1 + 127) << 23)) * __int_as_float((e2 + 127) << 23);
        }
    }
    if (tid == 0) fac[m] = __int_as_float((133 - a + 127) << 23);
}

// ---- host
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Workspace of the tensor-core path: X' [M, K] bf16 | S' [token tiles][G][128] fp32 | f [token tiles * 128].
size_t tc_ws(int64_t K, int64_t M) {
    const size_t Mt = static_cast<size_t>((M + kTcTok - 1) / kTcTok);
    const size_t G = static_cast<size_t>(K / 128);
    return align256(static_cast<size_t>(M) * static_cast<size_t>(K) * 2) + align256(Mt * G * kTcTok * 4) +
           align256(Mt * kTcTok * 4);
}

bool smem_ready(int dev) {
    static bool done[64] = {};
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return false;
    if (done[dev]) return true;
    if (cudaFuncSetAttribute(q4_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kTcSmem)) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    done[dev] = true;
    return true;
}

}  // namespace

bool q4i_prefill_tc_usable(int64_t K, int64_t M) {
    const char* v = std::getenv("Q4_PREFILL_TC");
    if (v && std::strcmp(v, "0") == 0) return false;
    if (K < 128 || K % 128 != 0 || K > 65536 || M < 1 || M > (1 << 24)) return false;
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return major == 10 && encoder() != nullptr;
}

size_t q4i_prefill_tc_ws(int64_t K, int64_t M) { return tc_ws(K, M); }

q4_status q4i_prefill_tc(const q4_matrix* W, const uint16_t* X, int64_t M, float* Y, void* ws, size_t ws_bytes,
                         cudaStream_t stream, bool pdl) {
    const int64_t K = W->K, N = W->N;
    if (ws_bytes < tc_ws(K, M)) return Q4_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || !smem_ready(dev)) return Q4_ERR_CUDA;
    const EncodeTiledFn enc = encoder();
    if (!enc) return Q4_ERR_CUDA;
    const int64_t Mt = (M + kTcTok - 1) / kTcTok;
    const int64_t RB = (N + kTcRows - 1) / kTcRows;
    if (RB * Mt > 0x7fffffffLL) return Q4_ERR_UNSUPPORTED_SHAPE;
    unsigned char* base = static_cast<unsigned char*>(ws);
    uint16_t* xp = reinterpret_cast<uint16_t*>(base);
    float* ssum = reinterpret_cast<float*>(base + align256(static_cast<size_t>(M) * K * 2));
    float* fac = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(ssum) +
                                          align256(static_cast<size_t>(Mt) * (K / 128) * kTcTok * 4));
    CUtensorMap map;
    std::memset(&map, 0, sizeof map);
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kTcTok)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, xp, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return Q4_ERR_CUDA;
    if (q4i_fault_injected()) return Q4_ERR_CUDA;

    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(Mt * kTcTok));
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, q4_tc_prep_kernel, X, static_cast<int>(K), static_cast<int>(M), xp, ssum, fac) !=
        cudaSuccess)
        return Q4_ERR_CUDA;

    TcParams tp;
    std::memset(&tp, 0, sizeof tp);
    tp.tiled = static_cast<const uint8_t*>(W->tiled);
    tp.ssum = ssum;
    tp.fac = fac;
    tp.y = Y;
    tp.N = static_cast<int>(N);
    tp.K = static_cast<int>(K);
    tp.M = static_cast<int>(M);
    tp.row_blocks = static_cast<int>(RB);
    cfg.gridDim = dim3(static_cast<unsigned>(RB * Mt));
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = kTcSmem;
    return cudaLaunchKernelEx(&cfg, q4_prefill_tc_kernel, map, tp) == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

int q4i_prefill_take_error() {
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_device_error, sizeof v) != cudaSuccess) return -1;
    if (v == 0) return 0;
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_tc_device_error, &zero, sizeof zero) != cudaSuccess) return -1;
    return 1;
}
