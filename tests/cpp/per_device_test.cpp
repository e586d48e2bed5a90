// Host test of attn_host::PerDevice (exact_attention_62_gb300/csrc/per_device.h),
// the per-device cache behind the library's launch set-up: built with g++ and
// run by tests/test_per_device.py, with a counting fake in place of the CUDA
// queries.  Exits non-zero on the first class of failure it finds.
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>

#include "per_device.h"

static int fails = 0;
#define CHECK(c)                                                   \
    do {                                                           \
        if (!(c)) {                                                \
            std::printf("FAIL line %d: %s\n", __LINE__, #c);       \
            ++fails;                                               \
        }                                                          \
    } while (0)

int main() {
    using attn_host::kMaxDevices;
    using attn_host::PerDevice;

    // Devices never share an entry, and each is set up exactly once.
    {
        PerDevice<int> c;
        int calls[4] = {0, 0, 0, 0};
        for (int rep = 0; rep < 3; ++rep)
            for (int d = 0; d < 4; ++d) {
                int v = 0;
                CHECK(c.get(d, &v, [&](int* o) {
                    ++calls[d];
                    *o = 100 + d;
                    return true;
                }));
                CHECK(v == 100 + d);
            }
        for (int d = 0; d < 4; ++d) CHECK(calls[d] == 1);
    }
    // A failed set-up is not cached: the next call retries, and a success
    // then stays.
    {
        PerDevice<int> c;
        int v = -1, calls = 0;
        CHECK(!c.get(2, &v, [&](int*) {
            ++calls;
            return false;
        }));
        CHECK(v == -1);
        CHECK(c.get(2, &v, [&](int* o) {
            ++calls;
            *o = 7;
            return true;
        }));
        CHECK(v == 7 && calls == 2);
        CHECK(c.get(2, &v, [&](int* o) {
            ++calls;
            *o = 8;
            return true;
        }));
        CHECK(v == 7 && calls == 2);
    }
    // Devices outside [0, kMaxDevices) get no value and no set-up.
    {
        PerDevice<int> c;
        int v = 0, calls = 0;
        auto make = [&](int* o) {
            ++calls;
            *o = 5;
            return true;
        };
        CHECK(!c.get(-1, &v, make));
        CHECK(!c.get(kMaxDevices, &v, make));
        CHECK(calls == 0);
        CHECK(c.get(kMaxDevices - 1, &v, make));
        CHECK(calls == 1 && v == 5);
    }
    // Sixteen threads asking for one device at once: one set-up, every
    // thread sees its value.
    {
        PerDevice<int> c;
        std::atomic<int> calls{0}, bad{0};
        std::vector<std::thread> ts;
        for (int t = 0; t < 16; ++t)
            ts.emplace_back([&] {
                int v = 0;
                const bool ok = c.get(3, &v, [&](int* o) {
                    calls++;
                    std::this_thread::yield();
                    *o = 42;
                    return true;
                });
                if (!ok || v != 42) bad++;
            });
        for (auto& t : ts) t.join();
        CHECK(calls == 1 && bad == 0);
    }
    std::printf(fails ? "per_device: %d failures\n" : "per_device: ok\n", fails);
    return fails ? 1 : 0;
}
