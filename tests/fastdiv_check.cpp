// Host check of the kernels' division by launch constants (FastDiv in
// kernels.h) against the division operator: edge and pseudo-random dividends in
// [0, 2^31) for every divisor given on the command line and a fixed set.
// Prints the number of mismatches (0 expected) and exits non-zero on any.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "kernels.h"

int main(int argc, char** argv) {
    std::vector<long long> divisors;
    for (int d = 1; d <= 1200; ++d) divisors.push_back(d);
    for (long long d : {1152LL, 4608LL, 8192LL, 9472LL, 32768LL, 75776LL, 131072LL, 65535LL, 65536LL, 65537LL,
                        (1LL << 20) + 1, (1LL << 30) - 1, 1LL << 30, (1LL << 30) + 1, (1LL << 31) - 1})
        divisors.push_back(d);
    for (int i = 1; i < argc; ++i) divisors.push_back(std::atoll(argv[i]));
    unsigned long long x = 0x9e3779b97f4a7c15ull;   // xorshift64 state
    long long bad = 0, checked = 0;
    for (long long d : divisors) {
        const xs::FastDiv f = xs::make_fastdiv(static_cast<int>(d));
        std::vector<long long> ns = {0, 1, 2, d - 1, d, d + 1, 2 * d - 1, 2 * d, (1LL << 31) - 1, (1LL << 31) - 2,
                                     ((1LL << 31) - 1) / d * d, ((1LL << 31) - 1) / d * d - 1};
        for (int k = 0; k < 2000; ++k) {
            x ^= x << 13;
            x ^= x >> 7;
            x ^= x << 17;
            ns.push_back(static_cast<long long>(x % (1ull << 31)));
            const long long m = static_cast<long long>(x >> 33) % 4096;   // near multiples of d
            ns.push_back(m * d - 1);
            ns.push_back(m * d);
        }
        for (long long n : ns) {
            if (n < 0 || n >= (1LL << 31)) continue;
            int q, r;
            xs::fdivmod(static_cast<int>(n), f, q, r);
            ++checked;
            if (q != n / d || r != n % d) {
                if (bad < 10) std::printf("d=%lld n=%lld: q=%d r=%d\n", d, n, q, r);
                ++bad;
            }
        }
    }
    std::printf("checked %lld mismatches %lld\n", checked, bad);
    return bad != 0;
}
