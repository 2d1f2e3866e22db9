// Checks gb300::fast_div (csrc/schedule.h) against the '/' operator: every
// divisor 1..5000 and, from there to 2^31 - 1, divisors near powers of two
// and pseudo-random ones, each against numerators at the edges (0, 1, the
// multiples of d around the top of the range and their neighbours, 2^31 - 1)
// and pseudo-random numerators.  Prints "ok <checks>" or the first mismatch.
#include <cstdint>
#include <cstdio>
#include <vector>

#include "schedule.h"

static uint64_t state = 0x9E3779B97F4A7C15ull;
static uint32_t next31() {   // xorshift64*, top 31 bits
    state ^= state >> 12;
    state ^= state << 25;
    state ^= state >> 27;
    return (uint32_t)((state * 2685821657736338717ull) >> 33);
}

int main() {
    const uint32_t top = 0x7FFFFFFFu;
    std::vector<uint32_t> divisors;
    for (uint32_t d = 1; d <= 5000; ++d) divisors.push_back(d);
    for (int l = 12; l <= 31; ++l) {
        const uint64_t p = uint64_t(1) << l;
        for (int64_t off = -3; off <= 3; ++off) {
            const int64_t d = (int64_t)p + off;
            if (d >= 1 && d <= (int64_t)top) divisors.push_back((uint32_t)d);
        }
    }
    for (int i = 0; i < 20000; ++i) divisors.push_back(next31() | 1u);
    uint64_t checks = 0;
    for (uint32_t d : divisors) {
        const gb300::FastDiv f = gb300::make_fastdiv(d);
        std::vector<uint32_t> xs = {0, 1, d - 1, d, d + 1, top, top - 1, top - d + 1};
        const uint32_t qmax = top / d;
        for (uint32_t q : {qmax, qmax - 1, qmax / 2 + 1}) {
            const uint64_t x = (uint64_t)q * d;
            for (int64_t off = -1; off <= 1; ++off) {
                const int64_t y = (int64_t)x + off;
                if (y >= 0 && y <= (int64_t)top) xs.push_back((uint32_t)y);
            }
        }
        for (int i = 0; i < 64; ++i) xs.push_back(next31());
        for (uint32_t x : xs) {
            if (x > top) continue;
            ++checks;
            if (gb300::fast_div(f, x) != x / d) {
                std::printf("mismatch x=%u d=%u got=%u want=%u\n", x, d, gb300::fast_div(f, x), x / d);
                return 1;
            }
        }
    }
    std::printf("ok %llu\n", (unsigned long long)checks);
    return 0;
}
