// map_cache.h -- a bounded cache of encoded TMA tensor maps.
//
// Every GEMM launch of the library needs a tensor map per operand shard, token
// chunk and output, and encoding one through the driver costs about a
// microsecond of host time: with the small layers (a few hundred tokens) that
// encoding, not the GPU, set the time of a step.  A map depends only on the
// arguments of the encoding (base address, element type, rank, extents, row
// strides, box, swizzle, L2 promotion), so it is cached under exactly those:
// a buffer at a new address (or of another shape) is a new key, and a cached
// map is never wrong for its key, even after the memory behind it was freed
// and reallocated.  The cache holds at most `capacity` maps; when it is full
// it is emptied and refills from the next calls.  A mutex guards it.
#pragma once

#include <cuda.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>

namespace tpmlp {
namespace abi {

struct MapKey {
    uint64_t ptr;
    uint64_t dims[3];
    uint64_t strides[2];  // bytes between consecutive indices of dims 1 and 2
    uint32_t box[3];
    uint32_t dtype, rank, swizzle, l2promo;
    uint32_t pad;  // keeps the key free of compiler padding (compared bytewise)
};
static_assert(sizeof(MapKey) == 8 + 24 + 16 + 12 + 16 + 4, "MapKey has no padding");

inline MapKey make_map_key(CUtensorMapDataType dtype, uint32_t rank, const void* ptr,
                           const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                           CUtensorMapSwizzle swizzle, CUtensorMapL2promotion l2promo) {
    MapKey k;
    std::memset(&k, 0, sizeof(k));
    k.ptr = reinterpret_cast<uint64_t>(ptr);
    for (uint32_t i = 0; i < rank && i < 3; ++i) {
        k.dims[i] = dims[i];
        k.box[i] = box[i];
        if (i + 1 < rank) k.strides[i] = strides[i];
    }
    k.dtype = static_cast<uint32_t>(dtype);
    k.rank = rank;
    k.swizzle = static_cast<uint32_t>(swizzle);
    k.l2promo = static_cast<uint32_t>(l2promo);
    return k;
}

struct MapKeyEq {
    bool operator()(const MapKey& a, const MapKey& b) const {
        return std::memcmp(&a, &b, sizeof(MapKey)) == 0;
    }
};

struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        // FNV-1a over the key's bytes
        const unsigned char* p = reinterpret_cast<const unsigned char*>(&k);
        uint64_t h = 1469598103934665603ULL;
        for (size_t i = 0; i < sizeof(MapKey); ++i) {
            h ^= p[i];
            h *= 1099511628211ULL;
        }
        return static_cast<size_t>(h);
    }
};

class MapCache {
  public:
    explicit MapCache(size_t capacity) : capacity_(capacity) {}

    // The map for `key`: from the cache, else from encode(out) (a callable
    // returning false on failure; failures are not cached).
    template <typename Encode>
    bool get(const MapKey& key, CUtensorMap* out, Encode&& encode) {
        {
            std::lock_guard<std::mutex> lk(mu_);
            auto it = maps_.find(key);
            if (it != maps_.end()) {
                *out = it->second;
                ++hits_;
                return true;
            }
        }
        if (!encode(out)) return false;
        std::lock_guard<std::mutex> lk(mu_);
        ++misses_;
        if (maps_.size() >= capacity_) maps_.clear();
        maps_.emplace(key, *out);
        return true;
    }

    void stats(uint64_t* hits, uint64_t* misses, uint64_t* entries) {
        std::lock_guard<std::mutex> lk(mu_);
        if (hits) *hits = hits_;
        if (misses) *misses = misses_;
        if (entries) *entries = maps_.size();
    }

    void clear() {
        std::lock_guard<std::mutex> lk(mu_);
        maps_.clear();
    }

  private:
    std::mutex mu_;
    size_t capacity_;
    uint64_t hits_ = 0, misses_ = 0;
    std::unordered_map<MapKey, CUtensorMap, MapKeyHash, MapKeyEq> maps_;
};

}  // namespace abi
}  // namespace tpmlp
