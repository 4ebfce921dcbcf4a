// Host-side checks of the static work partition in csrc/common.cuh (the helpers the decode
// and combine kernels share): every (unit, slot) is covered by exactly one CTA segment, the
// segment fields agree with the slot ranges, partial slots follow the first/last rule,
// cta_of_slot inverts cta_begin, and max_pieces_per_unit equals its per-unit definition
// (which counts exactly the CTAs with slots in a unit when no CTA range is empty).
// Exits non-zero on the first failure.
#include <cstdio>
#include <random>
#include <vector>

#include "common.cuh"

using namespace dsa;

#define CHECK(cond, ...)                                         \
    do {                                                         \
        if (!(cond)) {                                           \
            std::printf("FAIL %s: ", #cond);                     \
            std::printf(__VA_ARGS__);                            \
            std::printf("\n");                                   \
            return 1;                                            \
        }                                                        \
    } while (0)

int main() {
    std::mt19937_64 g(12345);
    const int64_t widths[] = {1, 2, 3, 64, 100, 384, 1000, 2048, 8192};
    for (int trial = 0; trial < 3000; ++trial) {
        const int64_t units = 1 + static_cast<int64_t>(g() % 300);
        const int64_t W = widths[g() % (sizeof(widths) / sizeof(widths[0]))];
        const int32_t groups = 1 + static_cast<int32_t>(g() % 3);
        const int32_t C = 1 + static_cast<int32_t>(g() % 400);
        Partition p;
        p.total_slots = units * W;
        p.width = static_cast<int32_t>(W);
        p.ctas = C;
        p.groups = groups;
        std::vector<uint8_t> covered(static_cast<size_t>(units * W), 0);
        std::vector<int32_t> ctas_in_unit(static_cast<size_t>(units), 0);
        for (int32_t c = 0; c < C; ++c) {
            const int64_t b = cta_begin(p, c), e = cta_begin(p, c + 1);
            CHECK(b <= e && e <= p.total_slots, "trial %d cta %d", trial, c);
            if (b < e) {
                CHECK(cta_of_slot(p, b) == c && cta_of_slot(p, e - 1) == c, "trial %d cta %d", trial, c);
            }
            int64_t first_unit = -1;
            const int32_t n = cta_segments(p, c, &first_unit);
            CHECK(n >= 0, "trial %d", trial);
            for (int32_t i = 0; i < n; ++i) {
                const Segment s = cta_segment(p, c, i);
                CHECK(s.unit == first_unit + i && s.unit < units, "trial %d", trial);
                CHECK(s.row == s.unit / groups && s.group == s.unit % groups, "trial %d", trial);
                CHECK(0 <= s.s0 && s.s0 < s.s1 && s.s1 <= W, "trial %d s0 %lld s1 %lld", trial,
                      static_cast<long long>(s.s0), static_cast<long long>(s.s1));
                CHECK(s.unit * W + s.s0 >= b && s.unit * W + s.s1 <= e, "trial %d", trial);
                const bool whole = s.s0 == 0 && s.s1 == W;
                CHECK(whole ? s.part == -1 : s.part == 2 * c + (i == 0 ? 0 : 1), "trial %d", trial);
                for (int64_t j = s.s0; j < s.s1; ++j) ++covered[static_cast<size_t>(s.unit * W + j)];
                ++ctas_in_unit[static_cast<size_t>(s.unit)];
            }
        }
        for (size_t x = 0; x < covered.size(); ++x) CHECK(covered[x] == 1, "trial %d slot %zu", trial, x);
        int32_t mp = 1;
        for (int32_t k : ctas_in_unit) mp = k > mp ? k : mp;
        int64_t by_def = 1;  // the definition, unit by unit (empty CTA ranges counted)
        for (int64_t u = 0; u < units; ++u) {
            const int64_t k = cta_of_slot(p, u * W + W - 1) - cta_of_slot(p, u * W) + 1;
            by_def = k > by_def ? k : by_def;
        }
        CHECK(max_pieces_per_unit(p) == by_def, "trial %d bound %lld definition %lld", trial,
              static_cast<long long>(max_pieces_per_unit(p)), static_cast<long long>(by_def));
        CHECK(by_def >= mp, "trial %d", trial);
        if (C <= p.total_slots) CHECK(by_def == mp, "trial %d: no empty ranges, so every piece has slots", trial);
    }
    std::printf("partition ok\n");
    return 0;
}
