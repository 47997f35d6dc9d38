// Host check of the tensor-core operand split (fa_split_bf16x3 in csrc/fa_internal.cuh, the
// function the operand-image kernel calls).  For floats over the whole range the span
// products use (random mantissas with exponents -149 ... 64, plus 0, 1, the largest float and
// the normal/subnormal boundary) it checks that
//   * x = p1 + p2 + p3 exactly (the parts added in double, which holds them exactly), except
//     for a subnormal third part, whose loss must stay below 2^-133;
//   * the parts are bf16 values: p1 keeps at most 8 significant bits of x, p2 at most 8 of
//     the remainder, p3 is what is left;
//   * for pairs (x, y) with x, y >= 2^-100, the six products the MMAs form,
//     p1q1 + p1q2 + p2q1 + p1q3 + p2q2 + p3q1 (each exact in double, their sum exact too),
//     are within 2^-21 of x*y relative -- the three dropped terms are each below 2^-22.
// Prints "ok N" (N checks) or the first failure, and exits non-zero on a failure.
#include <cmath>
#include <cstdio>
#include <random>
#include <vector>

#include "../constrained_decoding_diffusion_gb300/csrc/fa_internal.cuh"

static double part(uint32_t b) { return (double)fa_bits_f32(b << 16); }

static int sig_bits(double v) {   // significant bits of a double holding a float-sized value
    if (v == 0.0) return 0;
    int e;
    double m = std::frexp(std::fabs(v), &e);   // m in [0.5, 1)
    int n = 0;
    while (m != 0.0 && n < 60) {
        m = m * 2.0;
        m -= std::floor(m);
        ++n;
    }
    return n;
}

int main() {
    std::mt19937_64 rng(12345);
    std::vector<float> xs = {0.0f, 1.0f, 3.4028234663852886e38f, 1.1754943508222875e-38f, 1.1754942e-38f,
                             1.4e-45f, 0.99999994f, 1.0000001f};
    for (int i = 0; i < 200000; ++i) {
        const uint32_t mant = (uint32_t)(rng() & 0x7fffffu);
        const int e = (int)(rng() % 214) - 149;             // -149 ... 64
        float x;
        if (e < -126) x = fa_bits_f32(mant >> (-126 - e));   // subnormal
        else x = fa_bits_f32(((uint32_t)(e + 127) << 23) | mant);
        xs.push_back(x);
    }
    long checks = 0;
    std::vector<double> p1s(xs.size()), p2s(xs.size()), p3s(xs.size());
    for (size_t i = 0; i < xs.size(); ++i) {
        const float x = xs[i];
        uint32_t b1, b2, b3;
        fa_split_bf16x3(x, b1, b2, b3);
        const double p1 = part(b1), p2 = part(b2), p3 = part(b3), sum = p1 + p2 + p3;
        p1s[i] = p1, p2s[i] = p2, p3s[i] = p3;
        const double r2 = (double)x - p1 - p2;              // exact in double
        const bool r2_subnormal = r2 != 0.0 && std::fabs(r2) < std::ldexp(1.0, -126);
        const double loss = std::fabs(sum - (double)x);
        if (loss != 0.0 && !r2_subnormal) {
            printf("split not exact: x=%a p1=%a p2=%a p3=%a\n", x, p1, p2, p3);
            return 1;
        }
        if (loss > std::ldexp(1.0, -133)) {
            printf("split loses %a of x=%a\n", loss, x);
            return 1;
        }
        if (sig_bits(p1) > 8 || sig_bits(p2) > 8 || sig_bits(p3) > 8 || p1 < 0 || p2 < 0 || p3 < 0) {
            printf("parts not bf16: x=%a p1=%a p2=%a p3=%a\n", x, p1, p2, p3);
            return 1;
        }
        ++checks;
    }
    std::uniform_int_distribution<size_t> pick(0, xs.size() - 1);
    for (int i = 0; i < 200000; ++i) {
        const size_t a = pick(rng), b = pick(rng);
        const double x = xs[a], y = xs[b];
        if (x < std::ldexp(1.0, -100) || y < std::ldexp(1.0, -100)) continue;   // no subnormal parts
        const double six = p1s[a] * p1s[b] + p1s[a] * p2s[b] + p2s[a] * p1s[b] + p1s[a] * p3s[b] +
                           p2s[a] * p2s[b] + p3s[a] * p1s[b];
        const double rel = std::fabs(six - x * y) / (x * y);
        if (!(rel <= std::ldexp(1.0, -21))) {
            printf("six-term product off by %.3e (relative): x=%a y=%a\n", rel, x, y);
            return 1;
        }
        ++checks;
    }
    printf("ok %ld\n", checks);
    return 0;
}
