// cache.cu -- a bounded pool of device slots as a cache over every expert's
// packed blob in host memory (the pages' slot pool fed from storage, with a
// frequency-and-recency replacement: the xix.ai article, paragraphs on how it
// works; the agentlenshq article, how expert streaming works). Host code only:
// the policy decides which slot each (layer, expert) occupies; misses are
// copied host -> device with one cudaMemcpyAsync per blob (spread over a few
// copy streams forked from and joined back to the caller's stream, so several
// copy engines run at once) and the affected rows of the context's slot table
// are rewritten, so the GPU kernels see only
// resident experts through the same indirection as a fully resident pool.
// Results do not depend on where an expert sits, so a cached run is
// bit-identical to a fully resident one.
#include <cstring>
#include <new>
#include <set>
#include <tuple>
#include <vector>

#include "smoe_internal.h"

namespace smoe {

// Replacement policy: a slot holds one (layer, expert); on a miss the victim is
// the resident expert used least often, ties to the one used least recently,
// never one named by the current request. Free slots are used first.
class SlotPolicy {
public:
    struct Fill {
        int64_t slot;
        int32_t layer, expert;
    };

    SlotPolicy(int32_t n_layers, int32_t E, int64_t n_slots)
        : L_(n_layers), E_(E), S_(n_slots), map_(size_t(n_layers) * E, -1), owner_(n_slots, -1), freq_(n_slots, 0),
          last_(n_slots, 0), pin_(n_slots, 0), seen_(E, 0), placed_(n_slots, 0)
    {
        for (int64_t s = n_slots - 1; s >= 0; --s) free_.push_back(s);
    }

    int32_t slot_of(int32_t layer, int32_t e) const { return int32_t(map_[size_t(layer) * E_ + e]); }

    // Makes ids[0..n) of `layer` resident. Returns 0, or SMOE_EINVAL (bad id)
    // or SMOE_ENOMEM (more distinct experts than slots); on error nothing changes.
    int prepare(int32_t layer, const int32_t *ids, int32_t n, std::vector<Fill> &fills,
                std::vector<int64_t> &evicted, int32_t &hits, int32_t &misses)
    {
        fills.clear();
        evicted.clear();
        hits = misses = 0;
        if (layer < 0 || layer >= L_ || n < 0) return SMOE_EINVAL;
        for (int32_t i = 0; i < n; ++i)
            if (ids[i] < 0 || ids[i] >= E_) return SMOE_EINVAL;
        ++tick_;                                       // stamps: this request's experts and slots
        int64_t distinct = 0;
        for (int32_t i = 0; i < n; ++i)
            if (seen_[ids[i]] != tick_) {
                seen_[ids[i]] = tick_;
                ++distinct;
            }
        if (distinct > S_) return SMOE_ENOMEM;
        // pass 1: the resident ones are touched and pinned first, so no miss of
        // this request can evict an expert the request still needs
        for (int32_t i = 0; i < n; ++i) {
            const int64_t s = map_[size_t(layer) * E_ + ids[i]];
            if (s >= 0) {
                ++hits;
                touch(s);
                pin_[s] = tick_;
            }
        }
        // pass 2: misses (a repeated id is a hit once its first copy is placed)
        for (int32_t i = 0; i < n; ++i) {
            const size_t key = size_t(layer) * E_ + ids[i];
            if (map_[key] >= 0) {
                if (placed_[map_[key]] == tick_) {     // placed by an earlier occurrence in this request
                    ++hits;
                    touch(map_[key]);
                }
                continue;
            }
            ++misses;
            int64_t s;
            if (!free_.empty()) {
                s = free_.back();
                free_.pop_back();
            } else {
                auto it = order_.begin();
                while (pin_[std::get<2>(*it)] == tick_) ++it;   // a free one exists: distinct <= slots
                s = std::get<2>(*it);
                order_.erase(it);
                evicted.push_back(owner_[s]);
                map_[size_t(owner_[s])] = -1;
            }
            owner_[s] = int64_t(key);
            map_[key] = s;
            freq_[s] = 0;
            touch(s);
            pin_[s] = tick_;
            placed_[s] = tick_;
            fills.push_back({s, layer, ids[i]});
        }
        return SMOE_OK;
    }

private:
    void touch(int64_t s)
    {
        if (freq_[s] > 0) order_.erase(std::make_tuple(freq_[s], last_[s], s));
        ++freq_[s];
        last_[s] = tick_;
        order_.insert(std::make_tuple(freq_[s], last_[s], s));
    }

    int32_t L_, E_;
    int64_t S_;
    uint64_t tick_ = 0;
    std::vector<int64_t> map_;       // [L * E] slot or -1
    std::vector<int64_t> owner_;     // [S] layer * E + expert, or -1
    std::vector<uint64_t> freq_, last_;
    std::vector<uint64_t> pin_, seen_, placed_;  // request stamps (tick_): slot pinned, id seen, slot placed now
    std::vector<int64_t> free_;
    std::set<std::tuple<uint64_t, uint64_t, int64_t>> order_;   // (uses, last use, slot) of occupied slots
};

}  // namespace smoe

using smoe::SlotPolicy;

constexpr int kCopyStreams = 4;

struct smoe_cache {
    smoe_ctx *ctx;
    cudaStream_t side[kCopyStreams];   // the blob copies of one call, forked from and joined to its stream
    cudaEvent_t fork, join[kCopyStreams];
    const uint8_t *host_store;      // [n_layers][E][stride] packed blobs
    uint8_t *pool;                  // [n_slots][stride] device
    SlotPolicy *policy;
    int32_t *table_host;            // pinned mirror of the slot table [n_layers][E]
    uint64_t hits, misses, bytes;
    std::vector<SlotPolicy::Fill> fills;
    std::vector<int64_t> evicted;
};

extern "C" int smoe_cache_create(smoe_ctx *ctx, const void *host_store, uint64_t host_bytes, void *pool,
                                 uint64_t pool_bytes, void *stream, smoe_cache **out)
{
    if (!ctx || !host_store || !pool || !out) return SMOE_EINVAL;
    *out = nullptr;
    const uint64_t stride = ctx->layout.blob;
    const uint64_t n_experts = uint64_t(ctx->n_layers) * ctx->shape.E;
    if (host_bytes < n_experts * stride || pool_bytes < uint64_t(ctx->n_slots) * stride) return SMOE_ENOMEM;
    smoe_cache *c = new (std::nothrow) smoe_cache();
    if (!c) return SMOE_ENOMEM;
    c->ctx = ctx;
    c->host_store = static_cast<const uint8_t *>(host_store);
    c->pool = static_cast<uint8_t *>(pool);
    c->policy = new (std::nothrow) SlotPolicy(ctx->n_layers, ctx->shape.E, ctx->n_slots);
    if (!c->policy || cudaMallocHost(&c->table_host, n_experts * 4) != cudaSuccess) {
        delete c->policy;
        delete c;
        return SMOE_ENOMEM;
    }
    for (uint64_t i = 0; i < n_experts; ++i) c->table_host[i] = -1;   // nothing resident yet
    cudaError_t e = cudaEventCreateWithFlags(&c->fork, cudaEventDisableTiming);
    int made = 0;                                                    // streams and join events created
    for (; e == cudaSuccess && made < kCopyStreams; ++made) {
        e = cudaStreamCreateWithFlags(&c->side[made], cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->join[made], cudaEventDisableTiming);
        if (e != cudaSuccess) {
            if (c->side[made]) cudaStreamDestroy(c->side[made]);
            break;
        }
    }
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(ctx->table_dev, c->table_host, n_experts * 4, cudaMemcpyHostToDevice,
                            static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        for (int i = 0; i < made; ++i) {
            cudaStreamDestroy(c->side[i]);
            cudaEventDestroy(c->join[i]);
        }
        if (c->fork) cudaEventDestroy(c->fork);
        cudaFreeHost(c->table_host);
        delete c->policy;
        delete c;
        return SMOE_ECUDA;
    }
    *out = c;
    return SMOE_OK;
}

extern "C" int smoe_cache_destroy(smoe_cache *c)
{
    if (!c) return SMOE_OK;
    for (int i = 0; i < kCopyStreams; ++i) {          // released once their queued copies have run
        cudaStreamDestroy(c->side[i]);
        cudaEventDestroy(c->join[i]);
    }
    cudaEventDestroy(c->fork);
    cudaFreeHost(c->table_host);
    delete c->policy;
    delete c;
    return SMOE_OK;
}

extern "C" int smoe_cache_prepare(smoe_cache *c, int32_t layer, const int32_t *ids, int32_t n, void *stream,
                                  int32_t *hits, int32_t *misses)
{
    if (!c || (!ids && n > 0)) return SMOE_EINVAL;
    int32_t h = 0, m = 0;
    const int rc = c->policy->prepare(layer, ids, n, c->fills, c->evicted, h, m);
    if (rc) return rc;
    const smoe_ctx *ctx = c->ctx;
    const int32_t E = ctx->shape.E;
    const uint64_t stride = ctx->layout.blob;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    // The copies wait for everything queued on st before them (an evicted slot
    // may still be read by an earlier forward), run on up to kCopyStreams
    // streams, and st waits for all of them before the table rows change.
    const int nside = int(c->fills.size() < size_t(kCopyStreams) ? c->fills.size() : size_t(kCopyStreams));
    if (nside > 1) {
        e = cudaEventRecord(c->fork, st);
        for (int i = 0; i < nside && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(c->side[i], c->fork, 0);
    }
    for (size_t j = 0; j < c->fills.size() && e == cudaSuccess; ++j) {
        const SlotPolicy::Fill &f = c->fills[j];
        const uint8_t *src = c->host_store + (uint64_t(f.layer) * E + f.expert) * stride;
        e = cudaMemcpyAsync(c->pool + uint64_t(f.slot) * stride, src, stride, cudaMemcpyHostToDevice,
                            nside > 1 ? c->side[j % size_t(nside)] : st);
    }
    if (nside > 1)
        for (int i = 0; i < nside && e == cudaSuccess; ++i) {
            e = cudaEventRecord(c->join[i], c->side[i]);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(st, c->join[i], 0);
        }
    // the mirror, then the rows that changed: this layer's and those of evicted experts
    std::vector<int32_t> rows(1, layer);
    for (int64_t key : c->evicted) {
        const int32_t l = int32_t(key / E);
        c->table_host[key] = -1;
        bool seen = false;
        for (int32_t r : rows) seen = seen || r == l;
        if (!seen) rows.push_back(l);
    }
    for (const SlotPolicy::Fill &f : c->fills) c->table_host[uint64_t(f.layer) * E + f.expert] = int32_t(f.slot);
    for (int32_t r : rows)
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(ctx->table_dev + uint64_t(r) * E, c->table_host + uint64_t(r) * E, uint64_t(E) * 4,
                                cudaMemcpyHostToDevice, st);
    c->hits += uint64_t(h);
    c->misses += uint64_t(m);
    c->bytes += uint64_t(c->fills.size()) * stride;
    if (hits) *hits = h;
    if (misses) *misses = m;
    return e == cudaSuccess ? SMOE_OK : SMOE_ECUDA;
}

extern "C" int smoe_cache_stats(const smoe_cache *c, uint64_t *hits, uint64_t *misses, uint64_t *bytes_copied)
{
    if (!c) return SMOE_EINVAL;
    if (hits) *hits = c->hits;
    if (misses) *misses = c->misses;
    if (bytes_copied) *bytes_copied = c->bytes;
    return SMOE_OK;
}

extern "C" int smoe_cache_simulate(int32_t n_layers, int32_t E, int64_t n_slots, const int32_t *requests,
                                   int32_t n_requests, int32_t *out_slots, int64_t *hits, int64_t *misses)
{
    if (n_layers <= 0 || E <= 0 || n_slots <= 0 || n_requests < 0 || (n_requests > 0 && (!requests || !out_slots)))
        return SMOE_EINVAL;
    SlotPolicy pol(n_layers, E, n_slots);
    std::vector<SlotPolicy::Fill> fills;
    std::vector<int64_t> evicted;
    int64_t th = 0, tm = 0, o = 0, w = 0;
    for (int32_t r = 0; r < n_requests; ++r) {
        const int32_t layer = requests[o], n = requests[o + 1];
        const int32_t *ids = requests + o + 2;
        int32_t h = 0, m = 0;
        const int rc = pol.prepare(layer, ids, n, fills, evicted, h, m);
        if (rc) return rc;
        for (int32_t i = 0; i < n; ++i) out_slots[w++] = pol.slot_of(layer, ids[i]);
        th += h;
        tm += m;
        o += 2 + n;
    }
    if (hits) *hits = th;
    if (misses) *misses = tm;
    return SMOE_OK;
}
