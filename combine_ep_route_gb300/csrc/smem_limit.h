// smem_limit.h -- bookkeeping of the dynamic shared-memory limit raised per
// (kernel, device).
//
// A kernel that asks for more than 48 KiB of dynamic shared memory must first
// have its limit raised with cudaFuncSetAttribute, and that attribute belongs
// to the device current when it is set. Launchers call SmemLimits::ensure
// before every launch; it calls the raise function only when this (kernel,
// device) has not yet been raised to at least `bytes`, and records the new
// limit once the raise succeeds. A mutex makes it safe from several host
// threads driving several devices. Plain C++ (no CUDA types) so that its logic
// is testable on a machine without a GPU.
#pragma once

#include <cstddef>
#include <mutex>
#include <vector>

namespace ep {

class SmemLimits {
public:
    static constexpr size_t kDefaultLimit = 48 * 1024;

    // Returns 0 if nothing had to be done or `raise()` returned 0; otherwise
    // the non-zero value `raise()` returned (nothing is recorded then).
    template <class Raise>
    int ensure(const void *fn, int device, size_t bytes, Raise &&raise) {
        if (bytes <= kDefaultLimit) return 0;
        std::lock_guard<std::mutex> lock(mu_);
        Entry *e = find(fn, device);
        if (e && e->bytes >= bytes) return 0;
        const int rc = raise();
        if (rc != 0) return rc;
        if (e)
            e->bytes = bytes;
        else
            entries_.push_back(Entry{fn, device, bytes});
        return 0;
    }

    // The limit recorded for (fn, device), 0 if none.
    size_t recorded(const void *fn, int device) {
        std::lock_guard<std::mutex> lock(mu_);
        const Entry *e = find(fn, device);
        return e ? e->bytes : 0;
    }

private:
    struct Entry {
        const void *fn;
        int device;
        size_t bytes;
    };
    Entry *find(const void *fn, int device) {
        for (Entry &e : entries_)
            if (e.fn == fn && e.device == device) return &e;
        return nullptr;
    }
    std::mutex mu_;
    std::vector<Entry> entries_;
};

// The one table of the library (an inline function's static is shared by every
// translation unit of the shared object).
inline SmemLimits &smem_limits() {
    static SmemLimits table;
    return table;
}

}  // namespace ep
