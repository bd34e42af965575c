// Host side of libq4.so: the offline int4 export (q4_pack_host) and status strings.
//
// The export follows the rumik-oss-1 int4 engine page (rtts.neoandmatrix.me,
// "Step 3: an int4 file and a first kernel"): for every row, each run of 128
// columns carries one fp16 scale and one fp16 minimum; 4-bit codes packed in pairs.  The
// arithmetic is plain IEEE double; this file is compiled with
// -ffp-contract=off so no multiply-add is fused and the result is the same on
// x86-64 and aarch64 hosts.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <atomic>

#include "q4.h"

namespace {

// Round a double to IEEE binary16, nearest-even, working on the bit pattern.
// Sets *overflow when the rounded magnitude exceeds the largest finite half.
uint16_t half_bits_from_double(double v, bool* overflow) {
    uint64_t b;
    std::memcpy(&b, &v, sizeof b);
    const uint16_t sign = static_cast<uint16_t>((b >> 63) << 15);
    const int exp = static_cast<int>((b >> 52) & 0x7FF);
    const uint64_t frac = b & ((uint64_t(1) << 52) - 1);
    if (exp == 0x7FF) { *overflow = true; return sign | 0x7C00; }
    if (exp == 0) return sign;  // zero or a double subnormal: far below half's range
    const uint64_t sig = (uint64_t(1) << 52) | frac;  // value = sig * 2^(exp - 1075)
    int e16 = exp - 1023 + 15;                         // biased half exponent if normal
    if (e16 >= 1) {
        // keep 11 significant bits: drop 42
        uint64_t q = sig >> 42;
        const uint64_t rem = sig & ((uint64_t(1) << 42) - 1);
        const uint64_t half = uint64_t(1) << 41;
        if (rem > half || (rem == half && (q & 1))) ++q;
        if (q == 2048) { q = 1024; ++e16; }
        if (e16 >= 31) { *overflow = true; return sign | 0x7C00; }
        return static_cast<uint16_t>(sign | (e16 << 10) | (q - 1024));
    }
    // subnormal half: count units of 2^-24; value / 2^-24 = sig * 2^(exp - 1051)
    const int shift = 1051 - exp;  // >= 43 here
    if (shift >= 64) return sign;  // below 2^-25 after the implicit bit: rounds to zero
    uint64_t q = sig >> shift;
    const uint64_t rem = sig & ((uint64_t(1) << shift) - 1);
    const uint64_t half = uint64_t(1) << (shift - 1);
    if (rem > half || (rem == half && (q & 1))) ++q;
    return static_cast<uint16_t>(sign | q);  // q == 1024 is the smallest normal, 0x0400
}

double double_from_half_bits(uint16_t h) {
    const int e = (h >> 10) & 0x1F;
    const int f = h & 0x3FF;
    const double mag = (e == 0) ? std::ldexp(static_cast<double>(f), -24)
                                : std::ldexp(static_cast<double>(1024 + f), e - 25);
    return (h & 0x8000) ? -mag : mag;
}

// Quantise rows [r_begin, r_end).  Returns false on a non-finite weight or an
// fp16 overflow.
bool pack_rows(const float* w, int64_t K, int64_t r_begin, int64_t r_end,
               uint8_t* codes, uint16_t* scales, uint16_t* mins) {
    const int64_t G = K / 128;
    uint8_t c[128];
    for (int64_t n = r_begin; n < r_end; ++n) {
        const float* row = w + n * K;
        for (int64_t g = 0; g < G; ++g) {
            const float* grp = row + g * 128;
            double lo = grp[0], hi = grp[0];
            for (int j = 0; j < 128; ++j) {
                const double v = grp[j];
                if (!std::isfinite(v)) return false;
                lo = v < lo ? v : lo;
                hi = v > hi ? v : hi;
            }
            bool ovf = false;
            const uint16_t sbits = half_bits_from_double((hi - lo) / 15.0, &ovf);
            const uint16_t mbits = half_bits_from_double(lo, &ovf);
            if (ovf) return false;
            const double s = double_from_half_bits(sbits);
            const double m = double_from_half_bits(mbits);
            for (int j = 0; j < 128; ++j) {
                double q = 0.0;
                if (s > 0.0) {
                    q = std::nearbyint((static_cast<double>(grp[j]) - m) / s);  // ties to even
                    q = q < 0.0 ? 0.0 : (q > 15.0 ? 15.0 : q);
                }
                c[j] = static_cast<uint8_t>(q);
            }
            uint8_t* out = codes + n * (K / 2) + g * 64;
            for (int j = 0; j < 64; ++j) out[j] = static_cast<uint8_t>(c[2 * j] | (c[2 * j + 1] << 4));
            scales[n * G + g] = sbits;
            mins[n * G + g] = mbits;
        }
    }
    return true;
}

}  // namespace

namespace {
// The int8 output head (per-row symmetric, see q4.h): s = fp16(max |w| / 127), rounded once from
// double; code = clamp(nearbyint(w / s), -127, 127) with the stored scale (round-half-even);
// s == 0 gives code 0.  False for a non-finite weight or a scale that overflows fp16.
bool pack_rows8(const float* w, int64_t K, int64_t r0, int64_t r1, int8_t* codes, uint16_t* scales) {
    for (int64_t r = r0; r < r1; ++r) {
        const float* row = w + r * K;
        double mx = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double v = row[k];
            if (!std::isfinite(v)) return false;
            mx = std::fabs(v) > mx ? std::fabs(v) : mx;
        }
        bool ovf = false;
        const uint16_t sbits = half_bits_from_double(mx / 127.0, &ovf);
        if (ovf) return false;
        scales[r] = sbits;
        const double s = double_from_half_bits(sbits);
        int8_t* out = codes + r * K;
        for (int64_t k = 0; k < K; ++k) {
            double q = s == 0.0 ? 0.0 : std::nearbyint(static_cast<double>(row[k]) / s);
            q = q < -127.0 ? -127.0 : (q > 127.0 ? 127.0 : q);
            out[k] = static_cast<int8_t>(q);
        }
    }
    return true;
}
}  // namespace

extern "C" q4_status q8_pack_host(const float* w, int64_t N, int64_t K, int8_t* codes, uint16_t* scales,
                                  int n_threads) {
    if (!w || !codes || !scales || N <= 0) return Q4_ERR_INVALID_ARG;
    if (K <= 0 || K % 128 != 0) return Q4_ERR_UNSUPPORTED_SHAPE;
    int T = n_threads > 0 ? n_threads : static_cast<int>(std::thread::hardware_concurrency());
    if (T < 1) T = 1;
    if (static_cast<int64_t>(T) > N) T = static_cast<int>(N);
    std::atomic<bool> ok{true};
    std::vector<std::thread> pool;
    pool.reserve(T);
    for (int t = 0; t < T; ++t) {
        const int64_t a = N * t / T, b = N * (t + 1) / T;
        pool.emplace_back([=, &ok] {
            if (!pack_rows8(w, K, a, b, codes, scales)) ok = false;
        });
    }
    for (auto& th : pool) th.join();
    return ok ? Q4_OK : Q4_ERR_INVALID_ARG;
}

extern "C" q4_status q4_pack_host(const float* w, int64_t N, int64_t K,
                                  uint8_t* codes, uint16_t* scales, uint16_t* mins,
                                  int n_threads) {
    if (!w || !codes || !scales || !mins || N <= 0) return Q4_ERR_INVALID_ARG;
    if (K <= 0 || K % 128 != 0) return Q4_ERR_UNSUPPORTED_SHAPE;
    int T = n_threads > 0 ? n_threads : static_cast<int>(std::thread::hardware_concurrency());
    if (T < 1) T = 1;
    if (static_cast<int64_t>(T) > N) T = static_cast<int>(N);
    std::atomic<bool> ok{true};
    if (T == 1) {
        ok = pack_rows(w, K, 0, N, codes, scales, mins);
    } else {
        std::vector<std::thread> pool;
        pool.reserve(T);
        for (int t = 0; t < T; ++t) {
            const int64_t a = N * t / T, b = N * (t + 1) / T;
            pool.emplace_back([=, &ok] {
                if (!pack_rows(w, K, a, b, codes, scales, mins)) ok = false;
            });
        }
        for (auto& th : pool) th.join();
    }
    return ok ? Q4_OK : Q4_ERR_INVALID_ARG;
}

extern "C" const char* q4_status_string(q4_status s) {
    switch (s) {
        case Q4_OK: return "ok";
        case Q4_ERR_INVALID_ARG: return "invalid argument";
        case Q4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (K must be a positive multiple of 128, at most 65536)";
        case Q4_ERR_MISALIGNED: return "misaligned pointer";
        case Q4_ERR_WORKSPACE: return "workspace missing or too small";
        case Q4_ERR_CUDA: return "CUDA error";
        case Q4_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}
