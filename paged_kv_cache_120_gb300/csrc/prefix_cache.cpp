// Host prefix-cache block pool: chained block hashes, a doubly linked free
// queue with lazy eviction, and sequences whose tables share cached blocks.
//
// The bookkeeping follows "01 · PagedAttention 与 KV cache 块管理":
//  §4.2 the free queue is a doubly linked list through the blocks (O(1)
//       removal from the middle), head = evicted first;
//  §4.3 allocation pops the head and drops the popped block's cached hash
//       (lazy eviction); a cache hit "touches" the block (count + 1, and off
//       the free queue if it was there); freeing returns blocks whose count
//       reaches 0 to the head if they have no hash (LIFO reuse) and to the
//       tail if they do (FIFO, so cached blocks live longest), walking the
//       table in reverse so that a chain's tail is evicted before its head;
//  §4.4 a full block's hash chains the parent block's hash and the block's
//       token ids (SHA-256); matching runs from the first block and stops at
//       the first miss;
//  §4.5 a match covers at most num_tokens - 1 tokens (the last prompt token
//       is always recomputed); a request that cannot get its blocks changes
//       nothing;
//  §5   block 0 is the null block: never free, never handed out.
// Readings: the chain's root is 32 zero bytes; token ids are hashed as
// little-endian int32; a prompt's full blocks are recorded as cached when
// they are allocated (their K/V are written in the same step, before any
// other request can read them), a decode block when its last slot is
// reserved; if two blocks carry the same hash the first stays the lookup
// target.
//
// Like the plain allocator it only builds inputs (block tables and slots)
// for the device calls and never touches device memory.
#include <algorithm>
#include <array>
#include <atomic>
#include <chrono>
#include <climits>
#include <condition_variable>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <memory>
#include <mutex>
#include <thread>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

// ------------------------------------------------------------ SHA-256
// FIPS 180-4, section 6.2: eight 32-bit working variables, 64 rounds per
// 512-bit block, message padded with a 1 bit, zeros and the 64-bit length.
using Digest = std::array<uint8_t, 32>;

constexpr uint32_t kRound[64] = {
    0x428a2f98, 0x71374491, 0xb5c0fbcf, 0xe9b5dba5, 0x3956c25b, 0x59f111f1, 0x923f82a4, 0xab1c5ed5,
    0xd807aa98, 0x12835b01, 0x243185be, 0x550c7dc3, 0x72be5d74, 0x80deb1fe, 0x9bdc06a7, 0xc19bf174,
    0xe49b69c1, 0xefbe4786, 0x0fc19dc6, 0x240ca1cc, 0x2de92c6f, 0x4a7484aa, 0x5cb0a9dc, 0x76f988da,
    0x983e5152, 0xa831c66d, 0xb00327c8, 0xbf597fc7, 0xc6e00bf3, 0xd5a79147, 0x06ca6351, 0x14292967,
    0x27b70a85, 0x2e1b2138, 0x4d2c6dfc, 0x53380d13, 0x650a7354, 0x766a0abb, 0x81c2c92e, 0x92722c85,
    0xa2bfe8a1, 0xa81a664b, 0xc24b8b70, 0xc76c51a3, 0xd192e819, 0xd6990624, 0xf40e3585, 0x106aa070,
    0x19a4c116, 0x1e376c08, 0x2748774c, 0x34b0bcb5, 0x391c0cb3, 0x4ed8aa4a, 0x5b9cca4f, 0x682e6ff3,
    0x748f82ee, 0x78a5636f, 0x84c87814, 0x8cc70208, 0x90befffa, 0xa4506ceb, 0xbef9a3f7, 0xc67178f2};

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

inline uint32_t bswap32(uint32_t x)
{
    return (x >> 24) | ((x >> 8) & 0xff00u) | ((x << 8) & 0xff0000u) | (x << 24);
}

// One 512-bit block, given as its 16 big-endian words, into the eight
// working variables; the message schedule is kept as a rolling window of
// 16 words.
void sha256_compress(uint32_t st[8], const uint32_t m[16])
{
    uint32_t w[16];
    for (int t = 0; t < 16; ++t)
        w[t] = m[t];
    uint32_t a = st[0], b = st[1], c = st[2], d = st[3], e = st[4], f = st[5], g = st[6], h = st[7];
#pragma GCC unroll 64
    for (int t = 0; t < 64; ++t) {
        uint32_t wt = w[t & 15];
        if (t >= 16) {
            const uint32_t x = w[(t + 1) & 15], y = w[(t + 14) & 15];
            wt += (rotr(x, 7) ^ rotr(x, 18) ^ (x >> 3)) + w[(t + 9) & 15] + (rotr(y, 17) ^ rotr(y, 19) ^ (y >> 10));
            w[t & 15] = wt;
        }
        const uint32_t t1 = h + (rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25)) + ((e & f) ^ (~e & g)) + kRound[t] + wt;
        const uint32_t t2 = (rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22)) + ((a & b) ^ (a & c) ^ (b & c));
        h = g;
        g = f;
        f = e;
        e = d + t1;
        d = c;
        c = b;
        b = a;
        a = t1 + t2;
    }
    st[0] += a;
    st[1] += b;
    st[2] += c;
    st[3] += d;
    st[4] += e;
    st[5] += f;
    st[6] += g;
    st[7] += h;
}

// Hash of a full block: SHA-256(parent hash || token ids as little-endian
// int32). Every part of the message (and its padding: a 1 bit, zeros, the
// 64-bit big-endian bit length) is 4-byte aligned, so its big-endian words
// are formed directly: a parent word as read, a token byte-swapped.
Digest block_hash(const Digest &parent, const int32_t *tokens, int n)
{
    uint32_t st[8] = {0x6a09e667, 0xbb67ae85, 0x3c6ef372, 0xa54ff53a, 0x510e527f, 0x9b05688c, 0x1f83d9ab,
                      0x5be0cd19};
    uint32_t m[16];
    for (int i = 0; i < 8; ++i)
        m[i] = (uint32_t)parent[4 * i] << 24 | (uint32_t)parent[4 * i + 1] << 16 | (uint32_t)parent[4 * i + 2] << 8 |
               (uint32_t)parent[4 * i + 3];
    int used = 8;  // words of m filled
    for (int i = 0; i < n; ++i) {
        m[used++] = bswap32((uint32_t)tokens[i]);
        if (used == 16) {
            sha256_compress(st, m);
            used = 0;
        }
    }
    const uint64_t bits = (32 + 4 * (uint64_t)n) * 8;
    m[used++] = 0x80000000u;
    if (used > 14) {
        while (used < 16)
            m[used++] = 0;
        sha256_compress(st, m);
        used = 0;
    }
    while (used < 14)
        m[used++] = 0;
    m[14] = (uint32_t)(bits >> 32);
    m[15] = (uint32_t)bits;
    sha256_compress(st, m);
    Digest d;
    for (int i = 0; i < 8; ++i)
        for (int j = 0; j < 4; ++j)
            d[4 * i + j] = (uint8_t)(st[i] >> (24 - 8 * j));
    return d;
}

// Key of (parent hash, block tokens) in the digest memo: a multiply-xorshift
// mix of the 64-bit words; candidates are always verified in full.
uint64_t memo_key(const Digest &parent, const int32_t *tokens, int n)
{
    uint64_t h = 0x243f6a8885a308d3ull;
    auto mix = [&h](uint64_t w) {
        h = (h ^ w) * 0x9e3779b97f4a7c15ull;
        h ^= h >> 29;
    };
    for (int i = 0; i < 4; ++i) {
        uint64_t w;
        std::memcpy(&w, parent.data() + 8 * i, 8);
        mix(w);
    }
    for (int i = 0; i < n; ++i)
        mix((uint64_t)(uint32_t)tokens[i] | (uint64_t)i << 32);
    return h;
}

// Index from a 64-bit key to the blocks that carry it, allocation-free:
// open addressing with linear probing over 2^k >= 2 * num_blocks slots (so at
// most half full), each slot holding the first block of a chain threaded
// through next[] in insertion order. Several keys' worth of blocks never share
// a chain; callers compare the full identity along the chain.
class BlockIndex {
  public:
    void init(int num_blocks)
    {
        size_t cap = 16;
        while (cap < 2 * (size_t)num_blocks)
            cap <<= 1;
        mask_ = cap - 1;
        keys_.assign(cap, 0);
        head_.assign(cap, -1);
        next_.assign(num_blocks, -1);
    }
    // First block under key, or -1; then next(b) walks the chain.
    int32_t first(uint64_t key) const
    {
        const size_t i = find(key);
        return head_[i];
    }
    int32_t next(int32_t b) const { return next_[b]; }
    void insert(uint64_t key, int32_t b)
    {
        const size_t i = find(key);
        next_[b] = -1;
        if (head_[i] < 0) {
            keys_[i] = key;
            head_[i] = b;
            return;
        }
        int32_t t = head_[i];
        while (next_[t] >= 0)
            t = next_[t];
        next_[t] = b;
    }
    void erase(uint64_t key, int32_t b)
    {
        const size_t i = find(key);
        if (head_[i] == b) {
            head_[i] = next_[b];
            if (head_[i] < 0)
                remove_slot(i);
        } else {
            for (int32_t t = head_[i]; t >= 0; t = next_[t])
                if (next_[t] == b) {
                    next_[t] = next_[b];
                    break;
                }
        }
        next_[b] = -1;
    }

  private:
    // The slot holding key, or the empty slot where it would go.
    size_t find(uint64_t key) const
    {
        size_t i = key & mask_;
        while (head_[i] >= 0 && keys_[i] != key)
            i = (i + 1) & mask_;
        return i;
    }
    // Backward-shift deletion: later entries of the probe run whose home is
    // not cyclically within (hole, their slot] move into the hole.
    void remove_slot(size_t i)
    {
        size_t j = i;
        for (;;) {
            j = (j + 1) & mask_;
            if (head_[j] < 0)
                break;
            const size_t k = keys_[j] & mask_;
            const bool stays = i <= j ? (i < k && k <= j) : (i < k || k <= j);
            if (!stays) {
                keys_[i] = keys_[j];
                head_[i] = head_[j];
                i = j;
            }
        }
        head_[i] = -1;
    }
    size_t mask_ = 0;
    std::vector<uint64_t> keys_;
    std::vector<int32_t> head_, next_;
};

// Index key of a digest: its first 8 bytes (SHA-256 output is uniform).
uint64_t digest_key(const Digest &d)
{
    uint64_t x;
    std::memcpy(&x, d.data(), sizeof(x));
    return x;
}

// A small persistent pool: run(n, fn) calls fn(0..n-1) on the workers and
// the calling thread and returns when every call has finished. A worker
// polls for the next job for kPollUs after finishing one (admission waves
// come back to back; waking a sleeping thread costs tens of microseconds),
// then sleeps on a condition variable.
class WorkPool {
  public:
    explicit WorkPool(int threads)
    {
        for (int i = 0; i < threads; ++i)
            workers_.emplace_back([this] { loop(); });
    }
    ~WorkPool()
    {
        {
            std::lock_guard<std::mutex> l(m_);
            stop_ = true;
            stop_pub_.store(true, std::memory_order_release);
        }
        cv_.notify_all();
        for (auto &t : workers_)
            t.join();
    }
    void run(int n, const std::function<void(int)> &fn)
    {
        {
            std::lock_guard<std::mutex> l(m_);
            job_ = &fn;
            count_ = n;
            next_.store(0);
            done_ = 0;
            ++gen_;
            gen_pub_.store(gen_, std::memory_order_release);
        }
        cv_.notify_all();
        work();
        std::unique_lock<std::mutex> l(m_);
        done_cv_.wait(l, [&] { return done_ == count_; });
        job_ = nullptr;
    }

  private:
    void work()
    {
        for (;;) {
            const std::function<void(int)> *job;
            int count;
            {
                std::lock_guard<std::mutex> l(m_);
                job = job_;
                count = count_;
            }
            if (!job)
                return;
            const int i = next_.fetch_add(1);
            if (i >= count)
                return;
            (*job)(i);
            std::lock_guard<std::mutex> l(m_);
            if (++done_ == count_)
                done_cv_.notify_all();
        }
    }
    void loop()
    {
        uint64_t seen = 0;
        for (;;) {
            const auto t0 = std::chrono::steady_clock::now();
            while (gen_pub_.load(std::memory_order_acquire) == seen && !stop_pub_.load(std::memory_order_acquire) &&
                   std::chrono::steady_clock::now() - t0 < std::chrono::microseconds(kPollUs)) {
            }
            {
                std::unique_lock<std::mutex> l(m_);
                cv_.wait(l, [&] { return stop_ || gen_ != seen; });
                if (stop_)
                    return;
                seen = gen_;
            }
            work();
        }
    }
    std::vector<std::thread> workers_;
    std::mutex m_;
    std::condition_variable cv_, done_cv_;
    const std::function<void(int)> *job_ = nullptr;
    int count_ = 0, done_ = 0;
    std::atomic<int> next_{0};
    uint64_t gen_ = 0;
    bool stop_ = false;
    std::atomic<uint64_t> gen_pub_{0};  // gen_, readable without the lock
    std::atomic<bool> stop_pub_{false};
    static constexpr int kPollUs = 200;
};

// Hashing threads of a pool: PA_PCACHE_THREADS if set (0 = none), else
// min(16, hardware threads - 1).
int hash_threads()
{
    if (const char *e = std::getenv("PA_PCACHE_THREADS"))
        return std::max(0, std::min(64, std::atoi(e)));
    const int hw = (int)std::thread::hardware_concurrency();
    return std::max(0, std::min(16, hw - 1));
}

}  // namespace

struct pa_prefix_cache {
    int num_blocks = 0, block_size = 0;
    std::vector<int32_t> ref, prev, next;
    std::vector<char> in_free, hashed;
    std::vector<Digest> hash;
    int32_t head = -1, tail = -1, nfree = 0;
    // Recorded (cached) blocks by hash; among blocks with the same hash the
    // earliest recorded is the lookup target.
    BlockIndex cached;
    // Digest memo: a recorded block keeps its parent hash and token ids, so a
    // later (parent, tokens) pair equal to them reuses its hash instead of
    // running SHA-256 again. Only a full match of both is taken: the digest
    // is exactly the one SHA-256 would give.
    BlockIndex memo;
    std::vector<Digest> parent_of;
    std::vector<int32_t> tokens_of;  // block_size ids per block
    std::vector<uint64_t> memo_key_of;
    struct Seq {
        std::vector<int32_t> table, tokens;
        std::vector<Digest> hashes;
        bool cache = true;  // false: never matched against nor recorded
    };
    std::unordered_map<int, Seq> seqs;
    int next_id = 0;
    std::unique_ptr<WorkPool> pool;  // hashes a wave's requests in parallel (created on first use)
    bool pool_tried = false;

    // free queue
    void unlink(int32_t b)
    {
        (prev[b] >= 0 ? next[prev[b]] : head) = next[b];
        (next[b] >= 0 ? prev[next[b]] : tail) = prev[b];
        prev[b] = next[b] = -1;
        in_free[b] = 0;
        --nfree;
    }
    void push_head(int32_t b)
    {
        prev[b] = -1;
        next[b] = head;
        (head >= 0 ? prev[head] : tail) = b;
        head = b;
        in_free[b] = 1;
        ++nfree;
    }
    void push_tail(int32_t b)
    {
        next[b] = -1;
        prev[b] = tail;
        (tail >= 0 ? next[tail] : head) = b;
        tail = b;
        in_free[b] = 1;
        ++nfree;
    }
    // Digest of a full block: from the memo when a recorded block has the
    // same parent hash and token ids, else SHA-256.
    Digest digest(const Digest &parent, const int32_t *tokens) const
    {
        const int B = block_size;
        for (int32_t b = memo.first(memo_key(parent, tokens, B)); b >= 0; b = memo.next(b))
            if (parent_of[b] == parent &&
                std::memcmp(tokens_of.data() + (size_t)b * B, tokens, sizeof(int32_t) * (size_t)B) == 0)
                return hash[b];
        return block_hash(parent, tokens, B);
    }
    // The lookup target for a hash, or -1.
    int32_t lookup(const Digest &d) const
    {
        for (int32_t b = cached.first(digest_key(d)); b >= 0; b = cached.next(b))
            if (hash[b] == d)
                return b;
        return -1;
    }
    // cache
    void evict(int32_t b)
    {
        if (!hashed[b])
            return;
        memo.erase(memo_key_of[b], b);
        cached.erase(digest_key(hash[b]), b);
        hashed[b] = 0;
    }
    void record(int32_t b, const Digest &d, const Digest &parent, const int32_t *tokens)
    {
        hash[b] = d;
        hashed[b] = 1;
        cached.insert(digest_key(d), b);
        parent_of[b] = parent;
        std::memcpy(tokens_of.data() + (size_t)b * block_size, tokens, sizeof(int32_t) * (size_t)block_size);
        memo_key_of[b] = memo_key(parent, tokens, block_size);
        memo.insert(memo_key_of[b], b);
    }
    int32_t pop()
    {
        const int32_t b = head;
        unlink(b);
        evict(b);
        ref[b] = 1;
        return b;
    }
};

using pa::set_error;

namespace {

const pa_prefix_cache::Seq *find_seq(const pa_prefix_cache *c, int id)
{
    auto it = c->seqs.find(id);
    return it == c->seqs.end() ? nullptr : &it->second;
}

}  // namespace

extern "C" pa_prefix_cache *pa_pcache_create(int num_blocks, int block_size)
{
    if (num_blocks < 2 || block_size <= 0) {
        set_error(PA_ERR_INVALID_ARG, "pa_pcache_create: need num_blocks >= 2 (block 0 is the null block) "
                                      "and block_size > 0");
        return nullptr;
    }
    auto *c = new pa_prefix_cache();
    c->num_blocks = num_blocks;
    c->block_size = block_size;
    c->ref.assign(num_blocks, 0);
    c->prev.assign(num_blocks, -1);
    c->next.assign(num_blocks, -1);
    c->in_free.assign(num_blocks, 0);
    c->hashed.assign(num_blocks, 0);
    c->hash.assign(num_blocks, Digest{});
    c->parent_of.assign(num_blocks, Digest{});
    c->tokens_of.assign((size_t)num_blocks * block_size, 0);
    c->memo_key_of.assign(num_blocks, 0);
    c->cached.init(num_blocks);
    c->memo.init(num_blocks);
    for (int32_t b = 1; b < num_blocks; ++b)
        c->push_tail(b);
    return c;
}

extern "C" void pa_pcache_destroy(pa_prefix_cache *c) { delete c; }

extern "C" int pa_pcache_num_free(const pa_prefix_cache *c)
{
    if (!c)
        return set_error(PA_ERR_INVALID_ARG, "pa_pcache_num_free: null cache");
    return c->nfree;
}

namespace {

// One prompt into the pool (pa_pcache_add_seq's rules). With cache false the
// prompt neither matches nor records: every block is fresh and unhashed.
// Returns PA_OK or PA_ERR_OUT_OF_BLOCKS, the latter with the pool unchanged
// and no error text set.
// The chained hashes of a prompt's full blocks (reads the pool, writes
// nothing: safe to run for several prompts at once).
void chain_digests(const pa_prefix_cache *c, const int32_t *tokens, int num_tokens, std::vector<Digest> &out)
{
    const int B = c->block_size, full = num_tokens / B;
    out.clear();
    out.reserve(full);
    Digest parent{};
    for (int i = 0; i < full; ++i) {
        parent = c->digest(parent, tokens + (size_t)i * B);
        out.push_back(parent);
    }
}

// chain_digests of a prompt whose first `k` full blocks hold the same tokens
// as those of a prompt with hashes `base`: chained, those hashes are equal,
// so they are copied and hashing resumes after them.
void chain_digests_from(const pa_prefix_cache *c, const int32_t *tokens, int num_tokens,
                        const std::vector<Digest> &base, int k, std::vector<Digest> &out)
{
    const int B = c->block_size, full = num_tokens / B;
    out.assign(base.begin(), base.begin() + k);
    out.reserve(full);
    Digest parent = k > 0 ? base[k - 1] : Digest{};
    for (int i = k; i < full; ++i) {
        parent = c->digest(parent, tokens + (size_t)i * B);
        out.push_back(parent);
    }
}

// `pre`, if given, holds the prompt's chain_digests (computed beforehand).
// `prev`, if given, is the sequence admitted just before: while this
// prompt's chained hashes equal its hashes, the lookup target of each is the
// block `prev` holds at that index (it matched it, or recorded it as the
// first block with that hash), so no index lookup is needed.
int admit_one(pa_prefix_cache *c, const int32_t *tokens, int num_tokens, bool cache, int *seq_id,
              int *num_cached_tokens, int *need_out, int *avail_out, std::vector<Digest> *pre = nullptr,
              const pa_prefix_cache::Seq *prev = nullptr)
{
    const int B = c->block_size;
    const int full = cache ? num_tokens / B : 0, nblk = (num_tokens + B - 1) / B;
    std::vector<Digest> hashes;
    if (cache && pre)
        hashes = std::move(*pre);
    else if (cache)
        chain_digests(c, tokens, num_tokens, hashes);
    std::vector<int32_t> hits;
    hits.reserve(full);
    const int same = (prev && prev->cache) ? (int)std::min(prev->hashes.size(), hashes.size()) : 0;
    bool with_prev = same > 0;
    for (int i = 0; i < full; ++i) {
        if ((long long)(i + 1) * B > num_tokens - 1)
            break;
        int32_t b;
        if (with_prev && i < same && hashes[i] == prev->hashes[i]) {
            b = prev->table[i];
        } else {
            with_prev = false;  // chained: once they differ they differ from here on
            b = c->lookup(hashes[i]);
            if (b < 0)
                break;
        }
        hits.push_back(b);
    }
    int touched_free = 0;
    for (int32_t b : hits)
        touched_free += c->in_free[b] ? 1 : 0;
    const int need = nblk - (int)hits.size();
    if (need > c->nfree - touched_free) {
        *need_out = need;
        *avail_out = c->nfree - touched_free;
        return PA_ERR_OUT_OF_BLOCKS;
    }
    pa_prefix_cache::Seq s;
    s.table.reserve(nblk);
    for (int32_t b : hits) {
        if (c->in_free[b])
            c->unlink(b);
        ++c->ref[b];
        s.table.push_back(b);
    }
    for (int i = (int)hits.size(); i < nblk; ++i) {
        const int32_t b = c->pop();
        s.table.push_back(b);
        if (i < full)
            c->record(b, hashes[i], i ? hashes[i - 1] : Digest{}, tokens + (size_t)i * B);
    }
    s.tokens.assign(tokens, tokens + num_tokens);
    s.hashes = std::move(hashes);
    s.cache = cache;
    const int id = c->next_id++;
    c->seqs.emplace(id, std::move(s));
    *seq_id = id;
    *num_cached_tokens = (int)hits.size() * B;
    return PA_OK;
}

}  // namespace

extern "C" int pa_pcache_add_seq(pa_prefix_cache *c, const int32_t *tokens, int num_tokens, int *seq_id,
                                 int *num_cached_tokens)
{
    if (!c || !seq_id || !num_cached_tokens || num_tokens <= 0 || !tokens)
        return set_error(PA_ERR_INVALID_ARG, "pa_pcache_add_seq: bad arguments (num_tokens must be > 0)");
    int need = 0, avail = 0;
    const int r = admit_one(c, tokens, num_tokens, true, seq_id, num_cached_tokens, &need, &avail);
    if (r == PA_ERR_OUT_OF_BLOCKS)
        return set_error(PA_ERR_OUT_OF_BLOCKS, "pa_pcache_add_seq: need %d blocks, %d free", need, avail);
    return r;
}

extern "C" int pa_pcache_admit(pa_prefix_cache *c, const int32_t *tokens, const int64_t *cu_tokens, int n,
                               int flags, int max_blocks_per_seq, int32_t *seq_ids, int32_t *num_cached,
                               int32_t *cu_seqlens_q, int32_t *seq_lens, int32_t *slot_mapping,
                               int64_t slot_capacity, int32_t *block_tables)
{
    if (!c || n < 0 || !cu_tokens || max_blocks_per_seq <= 0 || (flags & ~PA_PCACHE_NO_CACHE) ||
        (n > 0 && (!tokens || !seq_ids || !num_cached || !cu_seqlens_q || !seq_lens || !slot_mapping ||
                   !block_tables)))
        return set_error(PA_ERR_INVALID_ARG, "pa_pcache_admit: bad arguments");
    const int B = c->block_size;
    if (cu_tokens[0] != 0)
        return set_error(PA_ERR_INVALID_ARG, "pa_pcache_admit: cu_tokens[0] must be 0");
    for (int r = 0; r < n; ++r) {
        const int64_t len = cu_tokens[r + 1] - cu_tokens[r];
        if (len <= 0 || len > INT32_MAX)
            return set_error(PA_ERR_INVALID_ARG, "pa_pcache_admit: request %d has %lld tokens", r, (long long)len);
        if ((len + B - 1) / B > max_blocks_per_seq)
            return set_error(PA_ERR_INVALID_ARG, "pa_pcache_admit: request %d needs %lld blocks > %d", r,
                             (long long)((len + B - 1) / B), max_blocks_per_seq);
    }
    if (n > 0 && cu_tokens[n] > slot_capacity)
        return set_error(PA_ERR_INVALID_ARG, "pa_pcache_admit: slot_capacity %lld < %lld prompt tokens",
                         (long long)slot_capacity, (long long)cu_tokens[n]);
    if (n > 0 && cu_tokens[n] > INT32_MAX)
        return set_error(PA_ERR_INVALID_ARG, "pa_pcache_admit: more than 2^31 - 1 prompt tokens");
    const bool cache = !(flags & PA_PCACHE_NO_CACHE);
    // Phase 1: every request's hash chain (reads only). The full blocks a
    // request shares token for token with request 0 from the start have
    // request 0's hashes: those (up to the longest such run) are chained
    // first, then every request hashes the rest of its chain in parallel,
    // request 0 included.
    std::vector<std::vector<Digest>> pre;
    if (cache && n > 1) {
        pre.resize(n);
        const int32_t *t0 = tokens;
        const int full0 = (int)(cu_tokens[1] / B);
        std::vector<int> common(n, 0);
        int shared = 0;  // longest run of leading full blocks another request shares with request 0
        for (int r = 1; r < n; ++r) {
            const int32_t *tr = tokens + cu_tokens[r];
            const int fr = (int)((cu_tokens[r + 1] - cu_tokens[r]) / B);
            int k = 0;
            while (k < fr && k < full0 &&
                   std::memcmp(tr + (size_t)k * B, t0 + (size_t)k * B, sizeof(int32_t) * (size_t)B) == 0)
                ++k;
            common[r] = k;
            shared = std::max(shared, k);
        }
        std::vector<Digest> head;  // request 0's first `shared` chained hashes
        chain_digests(c, t0, shared * B, head);
        auto one = [&](int r) {
            chain_digests_from(c, tokens + cu_tokens[r], (int)(cu_tokens[r + 1] - cu_tokens[r]), head,
                               r > 0 ? common[r] : shared, pre[r]);
        };
        if (!c->pool_tried) {
            c->pool_tried = true;
            const int t = hash_threads();
            if (t > 0)
                c->pool.reset(new WorkPool(t));
        }
        if (c->pool && n >= 4)
            c->pool->run(n, one);
        else
            for (int r = 0; r < n; ++r)
                one(r);
    }
    // Phase 2: match, allocate and record in request order.
    cu_seqlens_q[0] = 0;
    int32_t q = 0;
    int admitted = 0;
    const pa_prefix_cache::Seq *prev = nullptr;
    for (; admitted < n; ++admitted) {
        const int len = (int)(cu_tokens[admitted + 1] - cu_tokens[admitted]);
        int sid = 0, hit = 0, need = 0, avail = 0;
        if (admit_one(c, tokens + cu_tokens[admitted], len, cache, &sid, &hit, &need, &avail,
                      pre.empty() ? nullptr : &pre[admitted], prev) != PA_OK)
            break;
        prev = &c->seqs.find(sid)->second;  // element addresses survive later insertions
        const auto &table = prev->table;
        seq_ids[admitted] = sid;
        num_cached[admitted] = hit;
        seq_lens[admitted] = len;
        // Slots of the uncached tokens, block by block (no division per token).
        for (int j = hit / B, pos = hit; pos < len; ++j) {
            const int32_t base = table[j] * B;
            const int end = std::min(len, (j + 1) * B);
            for (int o = pos - j * B; pos < end; ++pos, ++o)
                slot_mapping[q++] = base + o;
        }
        cu_seqlens_q[admitted + 1] = q;
        int32_t *row = block_tables + (size_t)admitted * max_blocks_per_seq;
        for (int j = 0; j < max_blocks_per_seq; ++j)
            row[j] = j < (int)table.size() ? table[j] : -1;
    }
    return admitted;
}

extern "C" int pa_pcache_append_token(pa_prefix_cache *c, int seq_id, int32_t token, int32_t *slot)
{
    if (!c || !slot)
        return set_error(PA_ERR_INVALID_ARG, "pa_pcache_append_token: null argument");
    auto it = c->seqs.find(seq_id);
    if (it == c->seqs.end())
        return set_error(PA_ERR_NOT_FOUND, "pa_pcache_append_token: unknown sequence %d", seq_id);
    auto &s = it->second;
    const int B = c->block_size;
    const int pos = (int)s.tokens.size();
    if (pos % B == 0) {
        if (c->nfree == 0)
            return set_error(PA_ERR_OUT_OF_BLOCKS, "pa_pcache_append_token: no free block");
        s.table.push_back(c->pop());
    }
    s.tokens.push_back(token);
    if ((pos + 1) % B == 0 && s.cache) {
        const Digest parent = s.hashes.empty() ? Digest{} : s.hashes.back();
        const int32_t *blk = s.tokens.data() + (pos + 1 - B);
        const Digest d = c->digest(parent, blk);
        s.hashes.push_back(d);
        c->record(s.table[pos / B], d, parent, blk);
    }
    *slot = s.table[pos / B] * B + pos % B;
    return PA_OK;
}

extern "C" int pa_pcache_free_seq(pa_prefix_cache *c, int seq_id)
{
    if (!c)
        return set_error(PA_ERR_INVALID_ARG, "pa_pcache_free_seq: null cache");
    auto it = c->seqs.find(seq_id);
    if (it == c->seqs.end())
        return set_error(PA_ERR_NOT_FOUND, "pa_pcache_free_seq: unknown sequence %d", seq_id);
    const auto &t = it->second.table;
    for (auto r = t.rbegin(); r != t.rend(); ++r) {
        const int32_t b = *r;
        if (--c->ref[b] == 0)
            c->hashed[b] ? c->push_tail(b) : c->push_head(b);
    }
    c->seqs.erase(it);
    return PA_OK;
}

extern "C" int pa_pcache_free_seqs(pa_prefix_cache *c, const int32_t *seq_ids, int n)
{
    if (!c || n < 0 || (n > 0 && !seq_ids))
        return set_error(PA_ERR_INVALID_ARG, "pa_pcache_free_seqs: bad arguments");
    for (int i = 0; i < n; ++i)
        if (c->seqs.find(seq_ids[i]) == c->seqs.end())
            return set_error(PA_ERR_NOT_FOUND, "pa_pcache_free_seqs: unknown sequence %d", seq_ids[i]);
    std::vector<int32_t> ids(seq_ids, seq_ids + n);
    std::sort(ids.begin(), ids.end());
    if (std::adjacent_find(ids.begin(), ids.end()) != ids.end())
        return set_error(PA_ERR_INVALID_ARG, "pa_pcache_free_seqs: a sequence is listed twice");
    for (int i = 0; i < n; ++i) {
        const int r = pa_pcache_free_seq(c, seq_ids[i]);
        if (r != PA_OK)
            return r;
    }
    return PA_OK;
}

extern "C" int pa_pcache_seq_len(const pa_prefix_cache *c, int seq_id)
{
    if (!c)
        return set_error(PA_ERR_INVALID_ARG, "pa_pcache_seq_len: null cache");
    const auto *s = find_seq(c, seq_id);
    if (!s)
        return set_error(PA_ERR_NOT_FOUND, "pa_pcache_seq_len: unknown sequence %d", seq_id);
    return (int)s->tokens.size();
}

extern "C" int pa_pcache_block_tables(const pa_prefix_cache *c, const int *seq_ids, int n,
                                      int max_blocks_per_seq, int32_t *out)
{
    if (!c || (n > 0 && (!seq_ids || !out)) || n < 0 || max_blocks_per_seq <= 0)
        return set_error(PA_ERR_INVALID_ARG, "pa_pcache_block_tables: bad arguments");
    for (int i = 0; i < n; ++i) {
        const auto *s = find_seq(c, seq_ids[i]);
        if (!s)
            return set_error(PA_ERR_NOT_FOUND, "pa_pcache_block_tables: unknown sequence %d", seq_ids[i]);
        if ((int)s->table.size() > max_blocks_per_seq)
            return set_error(PA_ERR_INVALID_ARG, "pa_pcache_block_tables: sequence %d has %zu blocks > %d",
                             seq_ids[i], s->table.size(), max_blocks_per_seq);
        int32_t *row = out + (size_t)i * max_blocks_per_seq;
        for (int j = 0; j < max_blocks_per_seq; ++j)
            row[j] = j < (int)s->table.size() ? s->table[j] : -1;
    }
    return PA_OK;
}

extern "C" int pa_pcache_slots(const pa_prefix_cache *c, int seq_id, int first_pos, int n, int32_t *out)
{
    if (!c || n < 0 || first_pos < 0 || (n > 0 && !out))
        return set_error(PA_ERR_INVALID_ARG, "pa_pcache_slots: bad arguments");
    const auto *s = find_seq(c, seq_id);
    if (!s)
        return set_error(PA_ERR_NOT_FOUND, "pa_pcache_slots: unknown sequence %d", seq_id);
    if ((long long)first_pos + n > (long long)s->tokens.size())
        return set_error(PA_ERR_INVALID_ARG, "pa_pcache_slots: positions beyond the sequence");
    const int B = c->block_size;
    for (int i = 0; i < n; ++i) {
        const int pos = first_pos + i;
        out[i] = s->table[pos / B] * B + pos % B;
    }
    return PA_OK;
}

extern "C" int pa_pcache_free_queue(const pa_prefix_cache *c, int32_t *out, int capacity)
{
    if (!c || capacity < 0 || (capacity > 0 && !out))
        return set_error(PA_ERR_INVALID_ARG, "pa_pcache_free_queue: bad arguments");
    int k = 0;
    for (int32_t b = c->head; b >= 0; b = c->next[b]) {
        if (k < capacity)
            out[k] = b;
        ++k;
    }
    return k;
}

extern "C" int pa_pcache_ref_count(const pa_prefix_cache *c, int block)
{
    if (!c || block < 0 || block >= c->num_blocks)
        return set_error(PA_ERR_INVALID_ARG, "pa_pcache_ref_count: bad block");
    return c->ref[block];
}

extern "C" int pa_pcache_block_hash(const pa_prefix_cache *c, int block, uint8_t *out)
{
    if (!c || !out || block < 0 || block >= c->num_blocks)
        return set_error(PA_ERR_INVALID_ARG, "pa_pcache_block_hash: bad arguments");
    if (!c->hashed[block])
        return 0;
    std::memcpy(out, c->hash[block].data(), 32);
    return 1;
}
