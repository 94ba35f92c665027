// A small table of per-context values: the device address of a __device__
// array as seen from one CUDA context. The address of a module's global
// belongs to the context that loaded the module; a device reset destroys that
// context, and the next one can load the module elsewhere. Every CUDA context
// has a process-unique 64-bit ID (cuCtxGetId) that is never reused, so an
// entry keyed by the ID cannot be returned for a later context.
//
// Plain C++ (no CUDA types), so the host tests compile it on a CPU.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <mutex>

namespace pcp {

template <int kSlots>
class CtxTable {
   public:
    // The value stored for context `id`, or nullptr.
    void* find(uint64_t id) {
        std::lock_guard<std::mutex> lock(mu_);
        for (int i = 0; i < kSlots; ++i)
            if (used_[i] && ids_[i] == id) return vals_[i];
        return nullptr;
    }

    // Store `val` for context `id` (replacing its entry, else the oldest one
    // once all slots are taken: contexts that no longer exist are never looked up
    // again, so losing their entries costs nothing).
    void put(uint64_t id, void* val) {
        std::lock_guard<std::mutex> lock(mu_);
        for (int i = 0; i < kSlots; ++i)
            if (used_[i] && ids_[i] == id) {
                vals_[i] = val;
                return;
            }
        const int i = next_;
        next_ = (next_ + 1) % kSlots;
        used_[i] = true;
        ids_[i] = id;
        vals_[i] = val;
    }

   private:
    std::mutex mu_;
    bool used_[kSlots] = {};
    uint64_t ids_[kSlots] = {};
    void* vals_[kSlots] = {};
    int next_ = 0;
};

}  // namespace pcp
