// Host-only check of the (kernel, device) shared-memory limit table that the
// library's launchers use (combine_ep_route_gb300/csrc/smem_limit.h). A fake
// "raise" stands in for cudaFuncSetAttribute and counts its calls.
#include "../combine_ep_route_gb300/csrc/smem_limit.h"

#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>

#define CHECK(c)                                                   \
    do {                                                           \
        if (!(c)) {                                                \
            std::printf("FAILED line %d: %s\n", __LINE__, #c);     \
            return 1;                                              \
        }                                                          \
    } while (0)

int main() {
    ep::SmemLimits t;
    int k1 = 0, k2 = 0;   // two "kernels", told apart by address
    int calls = 0;
    auto ok = [&] { ++calls; return 0; };
    // at or below the default limit nothing is raised or recorded
    CHECK(t.ensure(&k1, 0, 48 * 1024, ok) == 0 && calls == 0 && t.recorded(&k1, 0) == 0);
    // first large launch raises once; the same or a smaller size does not raise again
    CHECK(t.ensure(&k1, 0, 100000, ok) == 0 && calls == 1 && t.recorded(&k1, 0) == 100000);
    CHECK(t.ensure(&k1, 0, 100000, ok) == 0 && calls == 1);
    CHECK(t.ensure(&k1, 0, 60000, ok) == 0 && calls == 1);
    // a larger size raises again
    CHECK(t.ensure(&k1, 0, 200000, ok) == 0 && calls == 2 && t.recorded(&k1, 0) == 200000);
    // another device of the same kernel is its own record
    CHECK(t.recorded(&k1, 1) == 0);
    CHECK(t.ensure(&k1, 1, 100000, ok) == 0 && calls == 3 && t.recorded(&k1, 1) == 100000);
    CHECK(t.recorded(&k1, 0) == 200000);
    // another kernel on device 0 too
    CHECK(t.ensure(&k2, 0, 100000, ok) == 0 && calls == 4);
    // a failed raise is returned and not recorded, so the next launch tries again
    auto fail = [&] { ++calls; return 7; };
    CHECK(t.ensure(&k2, 3, 90000, fail) == 7 && calls == 5 && t.recorded(&k2, 3) == 0);
    CHECK(t.ensure(&k2, 3, 90000, ok) == 0 && calls == 6 && t.recorded(&k2, 3) == 90000);

    // many threads over 4 devices x 2 kernels: each (kernel, device) raised exactly
    // once for its largest size if every thread asks for the same size
    ep::SmemLimits u;
    std::atomic<int> raised{0};
    std::vector<std::thread> th;
    for (int i = 0; i < 16; ++i)
        th.emplace_back([&, i] {
            for (int r = 0; r < 1000; ++r) {
                const void *fn = (r & 1) ? (const void *)&k1 : (const void *)&k2;
                u.ensure(fn, (i + r) % 4, 150000, [&] { raised.fetch_add(1); return 0; });
            }
        });
    for (auto &x : th) x.join();
    CHECK(raised.load() == 8);
    for (int d = 0; d < 4; ++d) CHECK(u.recorded(&k1, d) == 150000 && u.recorded(&k2, d) == 150000);
    // the library-wide table is a single object
    CHECK(&ep::smem_limits() == &ep::smem_limits());
    std::printf("ok\n");
    return 0;
}
