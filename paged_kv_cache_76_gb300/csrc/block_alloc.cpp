// Host block allocator of the paged KV cache (C ABI: pa_alloc_* in pa.h).
//
// Design ("2.1 PagedAttention" §9.1-§9.3, §3, §6):
//  * a global pool of physical blocks, each with a reference count (number of
//    Block Tables holding it);
//  * a free queue kept as an intrusive doubly linked list over block ids
//    (prev/next int32 arrays): pop from the head and removal from the middle
//    are O(1), as the free queue in §9.2 requires;
//  * per-sequence Block Tables that grow one block at a time, only when the
//    last block is full (§3: nothing is reserved ahead);
//  * sharing (many tables point at one block) and Copy-on-Write (§6);
//  * release in reverse order; zero-count blocks go to the head of the queue
//    in that order (the free_blocks rule of §9.3 for blocks without a prefix
//    hash), so the tail block of a finished request is reused first;
//  * automatic prefix caching (off by default): full blocks carry a chained
//    64-bit FNV-1a hash of their token ids, a hash -> block map finds them
//    again for a new request's prompt, freed hashed blocks go to the tail of
//    the queue, and a cached block loses its hash only when the queue hands
//    it out again ("Khám phá vLLM … phần 2", prefix caching);
//  * preemption by swapping (§7): a second pool of CPU blocks with its own
//    free queue; swap-out moves a request's blocks there (pairs for the
//    copy) and releases its GPU blocks as a free would, swap-in takes new GPU
//    blocks and returns the CPU ones.
// Every entry point validates first and mutates only once success is certain;
// the host memory an entry point needs is allocated before it mutates
// anything, and a failed allocation returns PA_ERR_HOST_MEMORY (pa_guarded).
#include <algorithm>
#include <cstdint>
#include <memory>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"
#include "pa_guard.h"

namespace {

struct Seq {
  std::vector<int32_t> blocks;
  int64_t num_tokens = 0;
  // prefix caching: salt, hash of the last full block (salt before the
  // first), token ids of the partial last block; hashable = ids known
  uint64_t salt = 0, parent = 0;
  std::vector<int32_t> pending;
  bool hashable = true;
  bool swapped = false;  // blocks are CPU (swap-pool) blocks
};

// Free queue of the swap pool: the same intrusive doubly linked list.
struct Queue {
  std::vector<int32_t> prev, next;
  int32_t head = -1, tail = -1, n = 0;
  void init(int32_t count) {
    prev.assign(count, -1);
    next.assign(count, -1);
    head = tail = -1;
    n = 0;
    for (int32_t b = 0; b < count; ++b) {
      prev[b] = tail;
      if (tail < 0) head = b; else next[tail] = b;
      tail = b;
      ++n;
    }
  }
  int32_t pop_front() {
    const int32_t b = head;
    head = next[b];
    if (head < 0) tail = -1; else prev[head] = -1;
    next[b] = -1;
    --n;
    return b;
  }
  void push_front(int32_t b) {
    next[b] = head;
    prev[b] = -1;
    if (head < 0) tail = b; else prev[head] = b;
    head = b;
    ++n;
  }
};

// 64-bit FNV-1a: for each byte, xor it into the state, then multiply by the prime.
constexpr uint64_t kFnvOffset = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;

inline uint64_t fnv_bytes(uint64_t h, uint64_t v, int nbytes) {  // v's low nbytes, little-endian
  for (int i = 0; i < nbytes; ++i) {
    h ^= (v >> (8 * i)) & 0xffu;
    h *= kFnvPrime;
  }
  return h;
}

uint64_t hash_block(uint64_t parent, const int32_t* tokens, int64_t n) {
  uint64_t h = fnv_bytes(kFnvOffset, parent, 8);
  for (int64_t i = 0; i < n; ++i) h = fnv_bytes(h, (uint32_t)tokens[i], 4);
  return h;
}

}  // namespace

struct pa_alloc {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> ref;
  std::vector<int32_t> prev, next;  // free-queue links, -1 = none
  std::vector<uint8_t> in_free;
  int32_t head = -1, tail = -1, num_free = 0;
  std::unordered_map<int, Seq> seqs;
  int64_t cow_copies = 0;
  int64_t alloc_failures = 0;
  // prefix caching
  bool caching = false;
  std::vector<uint64_t> hash;
  std::vector<uint8_t> has_hash;
  std::unordered_map<uint64_t, int32_t> cached;
  int64_t lookup_blocks = 0, hit_blocks = 0, evictions = 0;
  // swap pool (0 blocks: none)
  int32_t num_cpu_blocks = 0;
  Queue cpu;

  void push_back(int32_t b) {
    prev[b] = tail;
    next[b] = -1;
    if (tail < 0) head = b; else next[tail] = b;
    tail = b;
    in_free[b] = 1;
    ++num_free;
  }
  void push_front(int32_t b) {
    next[b] = head;
    prev[b] = -1;
    if (head < 0) tail = b; else prev[head] = b;
    head = b;
    in_free[b] = 1;
    ++num_free;
  }
  void unlink(int32_t b) {
    int32_t p = prev[b], n = next[b];
    if (p < 0) head = n; else next[p] = n;
    if (n < 0) tail = p; else prev[n] = p;
    prev[b] = next[b] = -1;
    in_free[b] = 0;
    --num_free;
  }
  // popleft: caller has checked num_free > 0
  int32_t pop_front() {
    int32_t b = head;
    unlink(b);
    return b;
  }
  // a block from the head of the queue for new use (refcount 0 -> 1); a
  // cached block leaves the cache here
  int32_t take() {
    const int32_t b = pop_front();
    if (has_hash[b]) {
      auto it = cached.find(hash[b]);
      if (it != cached.end() && it->second == b) cached.erase(it);
      has_hash[b] = 0;
      ++evictions;
    }
    ref[b] = 1;
    return b;
  }
  // touch: one more reference; a free block leaves the queue
  void touch(int32_t b) {
    if (ref[b] == 0 && in_free[b]) unlink(b);
    ref[b] += 1;
  }
  Seq* find(int id) {
    auto it = seqs.find(id);
    return it == seqs.end() ? nullptr : &it->second;
  }
  const Seq* find(int id) const {
    auto it = seqs.find(id);
    return it == seqs.end() ? nullptr : &it->second;
  }
};

static inline int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Slots for the next n tokens of s, taking blocks as the last one fills.
static int grow(pa_alloc* a, Seq* s, int n_tokens, int32_t* slots_out) {
  const int64_t bs = a->block_size;
  const int64_t cur = s->num_tokens;
  if (n_tokens > 0 && cur % bs != 0 && a->ref[s->blocks.back()] > 1) return PA_ERR_SHARED_BLOCK;
  if (cur + n_tokens > (int64_t)INT32_MAX) return PA_ERR_INVALID;
  const int64_t need = cdiv64(cur + n_tokens, bs) - (int64_t)s->blocks.size();
  if (need > a->num_free) {
    ++a->alloc_failures;
    return PA_ERR_NO_FREE_BLOCKS;
  }
  if (need > 0) s->blocks.reserve(s->blocks.size() + (size_t)need);  // may throw: before any change
  for (int64_t i = 0; i < need; ++i) s->blocks.push_back(a->take());
  if (slots_out) {
    for (int64_t t = cur; t < cur + n_tokens; ++t)
      slots_out[t - cur] = (int32_t)((int64_t)s->blocks[t / bs] * bs + t % bs);
  }
  s->num_tokens = cur + n_tokens;
  return PA_OK;
}

extern "C" {

int pa_alloc_create(int num_blocks, int block_size, const int32_t* initial_free_order, pa_alloc** out) {
  return pa_guarded([&]() -> int {
    if (!out || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID;
    *out = nullptr;
    if (initial_free_order) {
      std::vector<uint8_t> seen(num_blocks, 0);
      for (int i = 0; i < num_blocks; ++i) {
        int32_t b = initial_free_order[i];
        if (b < 0 || b >= num_blocks || seen[b]) return PA_ERR_INVALID;
        seen[b] = 1;
      }
    }
    std::unique_ptr<pa_alloc> a(new pa_alloc());
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->ref.assign(num_blocks, 0);
    a->prev.assign(num_blocks, -1);
    a->next.assign(num_blocks, -1);
    a->in_free.assign(num_blocks, 0);
    a->hash.assign(num_blocks, 0);
    a->has_hash.assign(num_blocks, 0);
    for (int i = 0; i < num_blocks; ++i) a->push_back(initial_free_order ? initial_free_order[i] : i);
    *out = a.release();
    return PA_OK;
  });
}

void pa_alloc_destroy(pa_alloc* a) { delete a; }

int pa_alloc_add_seq(pa_alloc* a, int seq_id) {
  return pa_guarded([&]() -> int {
    if (!a || seq_id < 0 || a->find(seq_id)) return PA_ERR_INVALID;
    a->seqs.emplace(seq_id, Seq());
    return PA_OK;
  });
}

int pa_alloc_append_slots(pa_alloc* a, int seq_id, int n_tokens, int32_t* slots_out) {
  return pa_guarded([&]() -> int {
    if (!a || n_tokens < 0) return PA_ERR_INVALID;
    Seq* s = a->find(seq_id);
    if (!s || s->swapped) return PA_ERR_INVALID;
    const int st = grow(a, s, n_tokens, slots_out);
    if (st == PA_OK && n_tokens > 0) {  // token ids unknown: nothing more is hashed
      s->hashable = false;
      s->pending.clear();
    }
    return st;
  });
}

int pa_alloc_share(pa_alloc* a, int dst_seq, int src_seq, int n_tokens) {
  return pa_guarded([&]() -> int {
    if (!a || dst_seq == src_seq) return PA_ERR_INVALID;
    Seq* d = a->find(dst_seq);
    Seq* s = a->find(src_seq);
    if (!d || !s || d->swapped || s->swapped || !d->blocks.empty() || d->num_tokens != 0) return PA_ERR_INVALID;
    if (n_tokens < 0 || n_tokens > s->num_tokens) return PA_ERR_INVALID;
    const int64_t nblk = cdiv64(n_tokens, a->block_size);
    d->blocks.assign(s->blocks.begin(), s->blocks.begin() + nblk);
    for (int32_t b : d->blocks) a->touch(b);
    d->num_tokens = n_tokens;
    // the hash chain continues into dst only from a full, hashed last block
    d->salt = s->salt;
    d->pending.clear();
    if (n_tokens == 0) {
      d->parent = s->salt;
      d->hashable = true;
    } else if (n_tokens % a->block_size == 0 && a->has_hash[d->blocks.back()]) {
      d->parent = a->hash[d->blocks.back()];
      d->hashable = true;
    } else {
      d->hashable = false;
    }
    return PA_OK;
  });
}

int pa_alloc_cow(pa_alloc* a, int seq_id, int logical_block, int32_t* src_dst_out) {
  if (!a || !src_dst_out) return PA_ERR_INVALID;
  Seq* s = a->find(seq_id);
  if (!s || s->swapped || logical_block < 0 || logical_block >= (int)s->blocks.size()) return PA_ERR_INVALID;
  const int32_t b = s->blocks[logical_block];
  if (a->ref[b] == 1) {
    src_dst_out[0] = src_dst_out[1] = b;
    return PA_OK;
  }
  if (a->num_free < 1) {
    ++a->alloc_failures;
    return PA_ERR_NO_FREE_BLOCKS;
  }
  const int32_t n = a->take();
  a->ref[b] -= 1;
  s->blocks[logical_block] = n;
  ++a->cow_copies;
  src_dst_out[0] = b;
  src_dst_out[1] = n;
  return PA_OK;
}

int pa_alloc_free_seq(pa_alloc* a, int seq_id) {
  return pa_guarded([&]() -> int {
    if (!a) return PA_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_INVALID;
    const std::vector<int32_t>& blocks = it->second.blocks;
    if (it->second.swapped) {  // swap-pool blocks back to that pool's head, last first
      for (int32_t c : blocks) a->cpu.push_front(c);
      a->seqs.erase(it);
      return PA_OK;
    }
    // reverse order: tail block first; zero-count blocks are prepended keeping
    // that order, i.e. pushed to the front from the last of them to the first
    // (blocks without a hash); blocks with a hash are appended at the tail in
    // release order, so they are evicted last and a request's first block last
    std::vector<int32_t> no_hash, with_hash;
    no_hash.reserve(blocks.size());
    with_hash.reserve(blocks.size());
    for (auto rit = blocks.rbegin(); rit != blocks.rend(); ++rit) {
      a->ref[*rit] -= 1;
      if (a->ref[*rit] == 0) (a->has_hash[*rit] ? with_hash : no_hash).push_back(*rit);
    }
    for (auto rit = no_hash.rbegin(); rit != no_hash.rend(); ++rit) a->push_front(*rit);
    for (int32_t b : with_hash) a->push_back(b);
    a->seqs.erase(it);
    return PA_OK;
  });
}

int pa_alloc_block_table(const pa_alloc* a, int seq_id, int32_t* out, int cap, int* n_out) {
  if (!a) return PA_ERR_INVALID;
  const Seq* s = a->find(seq_id);
  if (!s) return PA_ERR_INVALID;
  const int n = (int)s->blocks.size();
  if (n_out) *n_out = n;
  if (n > cap || (n > 0 && !out)) return PA_ERR_INVALID;
  std::copy(s->blocks.begin(), s->blocks.end(), out);
  return PA_OK;
}

int pa_alloc_build_tables(const pa_alloc* a, const int* seq_ids, int n, int32_t* out,
                          int max_blocks_per_seq, int32_t* lens_out) {
  if (!a || n < 0 || max_blocks_per_seq < 0 || (n > 0 && (!seq_ids || !out))) return PA_ERR_INVALID;
  for (int i = 0; i < n; ++i) {
    const Seq* s = a->find(seq_ids[i]);
    if (!s || s->swapped || (int64_t)s->blocks.size() > max_blocks_per_seq || s->num_tokens > INT32_MAX)
      return PA_ERR_INVALID;
  }
  for (int i = 0; i < n; ++i) {
    const Seq* s = a->find(seq_ids[i]);
    int32_t* row = out + (int64_t)i * max_blocks_per_seq;
    std::copy(s->blocks.begin(), s->blocks.end(), row);
    std::fill(row + s->blocks.size(), row + max_blocks_per_seq, -1);
    if (lens_out) lens_out[i] = (int32_t)s->num_tokens;
  }
  return PA_OK;
}

int pa_alloc_common_prefix(const pa_alloc* a, const int* seq_ids, int n, int* n_blocks_out) {
  if (!a || n <= 0 || !seq_ids || !n_blocks_out) return PA_ERR_INVALID;
  const Seq* first = a->find(seq_ids[0]);
  if (!first || first->swapped) return PA_ERR_INVALID;
  int64_t common = first->num_tokens / a->block_size;  // full blocks only
  for (int i = 1; i < n; ++i) {
    const Seq* s = a->find(seq_ids[i]);
    if (!s || s->swapped) return PA_ERR_INVALID;
    common = std::min<int64_t>(common, s->num_tokens / a->block_size);
    int64_t k = 0;
    while (k < common && s->blocks[k] == first->blocks[k]) ++k;
    common = k;
  }
  *n_blocks_out = (int)common;
  return PA_OK;
}

int pa_alloc_seq_len(const pa_alloc* a, int seq_id, int64_t* n_tokens_out) {
  if (!a || !n_tokens_out) return PA_ERR_INVALID;
  const Seq* s = a->find(seq_id);
  if (!s) return PA_ERR_INVALID;
  *n_tokens_out = s->num_tokens;
  return PA_OK;
}

int pa_alloc_num_free(const pa_alloc* a) { return a ? a->num_free : PA_ERR_INVALID; }

int pa_alloc_ref(const pa_alloc* a, int block_id) {
  if (!a || block_id < 0 || block_id >= a->num_blocks) return PA_ERR_INVALID;
  return a->ref[block_id];
}

int pa_alloc_free_list(const pa_alloc* a, int32_t* out, int cap) {
  if (!a || cap < a->num_free || (a->num_free > 0 && !out)) return PA_ERR_INVALID;
  int i = 0;
  for (int32_t b = a->head; b >= 0; b = a->next[b]) out[i++] = b;
  return i;
}

int pa_alloc_get_stats(const pa_alloc* a, pa_alloc_stats* out) {
  if (!a || !out) return PA_ERR_INVALID;
  pa_alloc_stats st{};
  st.num_blocks = a->num_blocks;
  st.num_free = a->num_free;
  for (int32_t r : a->ref) {
    if (r > 0) ++st.num_used;
    if (r > 1) ++st.num_shared;
  }
  st.num_seqs = (int64_t)a->seqs.size();
  st.cow_copies = a->cow_copies;
  st.alloc_failures = a->alloc_failures;
  for (const auto& kv : a->seqs)
    st.waste_slots += (int64_t)kv.second.blocks.size() * a->block_size - kv.second.num_tokens;
  *out = st;
  return PA_OK;
}

int pa_alloc_enable_swap(pa_alloc* a, int num_cpu_blocks) {
  return pa_guarded([&]() -> int {
    if (!a || num_cpu_blocks <= 0 || a->num_cpu_blocks > 0) return PA_ERR_INVALID;
    a->num_cpu_blocks = num_cpu_blocks;
    a->cpu.init(num_cpu_blocks);
    return PA_OK;
  });
}

int pa_alloc_num_free_cpu(const pa_alloc* a) { return a ? a->cpu.n : PA_ERR_INVALID; }

int pa_alloc_is_swapped(const pa_alloc* a, int seq_id) {
  if (!a) return PA_ERR_INVALID;
  const Seq* s = a->find(seq_id);
  return s ? (s->swapped ? 1 : 0) : PA_ERR_INVALID;
}

int pa_alloc_swap_out(pa_alloc* a, int seq_id, int32_t* pairs_out, int cap, int* n_out) {
  return pa_guarded([&]() -> int {
    if (!a || a->num_cpu_blocks <= 0) return PA_ERR_INVALID;
    Seq* s = a->find(seq_id);
    if (!s || s->swapped) return PA_ERR_INVALID;
    const int n = (int)s->blocks.size();
    if (n_out) *n_out = n;
    if (n > cap || (n > 0 && !pairs_out)) return PA_ERR_INVALID;
    if (n > a->cpu.n) {
      ++a->alloc_failures;
      return PA_ERR_NO_FREE_BLOCKS;
    }
    std::vector<int32_t> cpu_blocks(n), no_hash, with_hash;
    no_hash.reserve(n);
    with_hash.reserve(n);
    for (int i = 0; i < n; ++i) {
      cpu_blocks[i] = a->cpu.pop_front();
      pairs_out[2 * i] = s->blocks[i];
      pairs_out[2 * i + 1] = cpu_blocks[i];
    }
    // release the GPU blocks exactly as pa_alloc_free_seq does
    for (auto rit = s->blocks.rbegin(); rit != s->blocks.rend(); ++rit) {
      a->ref[*rit] -= 1;
      if (a->ref[*rit] == 0) (a->has_hash[*rit] ? with_hash : no_hash).push_back(*rit);
    }
    for (auto rit = no_hash.rbegin(); rit != no_hash.rend(); ++rit) a->push_front(*rit);
    for (int32_t b : with_hash) a->push_back(b);
    s->blocks = std::move(cpu_blocks);
    s->swapped = true;
    return PA_OK;
  });
}

int pa_alloc_swap_in(pa_alloc* a, int seq_id, int32_t* pairs_out, int cap, int* n_out) {
  return pa_guarded([&]() -> int {
    if (!a) return PA_ERR_INVALID;
    Seq* s = a->find(seq_id);
    if (!s || !s->swapped) return PA_ERR_INVALID;
    const int n = (int)s->blocks.size();
    if (n_out) *n_out = n;
    if (n > cap || (n > 0 && !pairs_out)) return PA_ERR_INVALID;
    if (n > a->num_free) {
      ++a->alloc_failures;
      return PA_ERR_NO_FREE_BLOCKS;
    }
    std::vector<int32_t> gpu_blocks(n);
    for (int i = 0; i < n; ++i) {
      gpu_blocks[i] = a->take();
      pairs_out[2 * i] = s->blocks[i];
      pairs_out[2 * i + 1] = gpu_blocks[i];
    }
    for (int32_t c : s->blocks) a->cpu.push_front(c);  // last block ends at the head
    s->blocks = std::move(gpu_blocks);
    s->swapped = false;
    return PA_OK;
  });
}

uint64_t pa_block_hash(uint64_t parent, const int32_t* tokens, int n) {
  return hash_block(parent, tokens, (tokens && n > 0) ? n : 0);
}

int pa_alloc_enable_prefix_caching(pa_alloc* a) {
  if (!a) return PA_ERR_INVALID;
  a->caching = true;
  return PA_OK;
}

int pa_alloc_add_seq_cached(pa_alloc* a, int seq_id, const int32_t* tokens, int n_tokens, uint64_t salt,
                            int* n_cached_out) {
  return pa_guarded([&]() -> int {
    if (!a || seq_id < 0 || a->find(seq_id) || n_tokens < 0 || (n_tokens > 0 && !tokens)) return PA_ERR_INVALID;
    const int64_t bs = a->block_size;
    // longest run of cached prompt blocks, looked up in order (nothing changes yet)
    std::vector<int32_t> hits;
    uint64_t parent = salt;
    if (a->caching && n_tokens > 0) {
      const int64_t nfull = (int64_t)(n_tokens - 1) / bs;  // leave >= 1 token to compute
      for (int64_t i = 0; i < nfull; ++i) {
        const uint64_t h = hash_block(parent, tokens + i * bs, bs);
        ++a->lookup_blocks;
        auto it = a->cached.find(h);
        if (it == a->cached.end()) break;
        hits.push_back(it->second);
        parent = h;
      }
    }
    a->hit_blocks += (int64_t)hits.size();
    Seq sq;
    sq.salt = salt;
    sq.parent = parent;
    sq.blocks = hits;
    sq.num_tokens = (int64_t)hits.size() * bs;
    a->seqs.emplace(seq_id, std::move(sq));  // may throw: before any block changes hands
    for (int32_t b : hits) a->touch(b);
    if (n_cached_out) *n_cached_out = (int)(hits.size() * bs);
    return PA_OK;
  });
}

int pa_alloc_append_tokens(pa_alloc* a, int seq_id, const int32_t* tokens, int n_tokens, int32_t* slots_out) {
  return pa_guarded([&]() -> int {
    if (!a || n_tokens < 0 || (n_tokens > 0 && !tokens)) return PA_ERR_INVALID;
    Seq* s = a->find(seq_id);
    if (!s || s->swapped) return PA_ERR_INVALID;
    const int64_t first = s->num_tokens;
    const int st = grow(a, s, n_tokens, slots_out);
    if (st != PA_OK || !s->hashable) return st;
    // register every block these tokens fill (unless its hash is already
    // cached).  The slots are taken at this point, so a failed host allocation
    // here only ends the sequence's caching (it stays correct, uncached).
    const int64_t bs = a->block_size;
    try {
      for (int i = 0; i < n_tokens; ++i) {
        s->pending.push_back(tokens[i]);
        if ((int64_t)s->pending.size() == bs) {
          const uint64_t h = hash_block(s->parent, s->pending.data(), bs);
          const int32_t b = s->blocks[(first + i) / bs];
          if (a->caching && a->cached.find(h) == a->cached.end()) {
            a->cached.emplace(h, b);
            a->hash[b] = h;
            a->has_hash[b] = 1;
          }
          s->parent = h;
          s->pending.clear();
        }
      }
    } catch (const std::bad_alloc&) {
      s->hashable = false;
      s->pending.clear();
    }
    return PA_OK;
  });
}

int pa_alloc_block_hash(const pa_alloc* a, int block_id, uint64_t* hash_out, int* is_cached_out) {
  if (!a || block_id < 0 || block_id >= a->num_blocks || !is_cached_out) return PA_ERR_INVALID;
  *is_cached_out = a->has_hash[block_id] ? 1 : 0;
  if (hash_out) *hash_out = a->has_hash[block_id] ? a->hash[block_id] : 0;
  return PA_OK;
}

int pa_alloc_get_prefix_cache_stats(const pa_alloc* a, pa_prefix_cache_stats* out) {
  if (!a || !out) return PA_ERR_INVALID;
  out->lookup_blocks = a->lookup_blocks;
  out->hit_blocks = a->hit_blocks;
  out->evictions = a->evictions;
  out->cached_blocks = (int64_t)a->cached.size();
  return PA_OK;
}

// ---------------------------------------------------------------- checkpoint
// The whole allocator as a flat list of int64 words (layout in include/pa.h);
// map-ordered parts (sequences, cached hashes) are written in key order so
// that equal states give equal words.
namespace {
constexpr int64_t kExportMagic = 0x504b5641ll;  // "PKVA"
constexpr int64_t kExportVersion = 1;
}  // namespace

int pa_alloc_export(const pa_alloc* a, int64_t* out, int64_t cap, int64_t* n_out) {
  return pa_guarded([&]() -> int {
    if (!a || !n_out || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID;
    std::vector<int64_t> w;
    w.reserve(16 + 4 * (size_t)a->num_blocks);
    w.push_back(kExportMagic);
    w.push_back(kExportVersion);
    w.push_back(a->num_blocks);
    w.push_back(a->block_size);
    w.push_back(a->caching ? 1 : 0);
    w.push_back(a->num_cpu_blocks);
    w.push_back(a->cow_copies);
    w.push_back(a->alloc_failures);
    w.push_back(a->lookup_blocks);
    w.push_back(a->hit_blocks);
    w.push_back(a->evictions);
    w.push_back(a->num_free);
    for (int32_t b = a->head; b >= 0; b = a->next[b]) w.push_back(b);
    for (int32_t b = 0; b < a->num_blocks; ++b) w.push_back(a->ref[b]);
    for (int32_t b = 0; b < a->num_blocks; ++b) w.push_back(a->has_hash[b]);
    for (int32_t b = 0; b < a->num_blocks; ++b) w.push_back((int64_t)a->hash[b]);
    std::vector<std::pair<uint64_t, int32_t>> cached(a->cached.begin(), a->cached.end());
    std::sort(cached.begin(), cached.end());
    w.push_back((int64_t)cached.size());
    for (const auto& kv : cached) {
      w.push_back((int64_t)kv.first);
      w.push_back(kv.second);
    }
    w.push_back(a->num_cpu_blocks > 0 ? a->cpu.n : 0);
    if (a->num_cpu_blocks > 0)
      for (int32_t b = a->cpu.head; b >= 0; b = a->cpu.next[b]) w.push_back(b);
    std::vector<int> ids;
    ids.reserve(a->seqs.size());
    for (const auto& kv : a->seqs) ids.push_back(kv.first);
    std::sort(ids.begin(), ids.end());
    w.push_back((int64_t)ids.size());
    for (int id : ids) {
      const Seq& q = a->seqs.at(id);
      w.push_back(id);
      w.push_back(q.num_tokens);
      w.push_back((int64_t)q.salt);
      w.push_back((int64_t)q.parent);
      w.push_back(q.hashable ? 1 : 0);
      w.push_back(q.swapped ? 1 : 0);
      w.push_back((int64_t)q.blocks.size());
      for (int32_t b : q.blocks) w.push_back(b);
      w.push_back((int64_t)q.pending.size());
      for (int32_t t : q.pending) w.push_back(t);
    }
    *n_out = (int64_t)w.size();
    if (cap < (int64_t)w.size()) return cap == 0 && !out ? PA_OK : PA_ERR_INVALID;
    std::copy(w.begin(), w.end(), out);
    return PA_OK;
  });
}

int pa_alloc_import(const int64_t* words, int64_t n, pa_alloc** out) {
  return pa_guarded([&]() -> int {
    if (!words || n <= 0 || !out) return PA_ERR_INVALID;
    *out = nullptr;
    int64_t i = 0;
    bool bad = false;
    auto next = [&](int64_t lo, int64_t hi) -> int64_t {  // next word, required in [lo, hi]
      if (bad || i >= n) {
        bad = true;
        return lo;
      }
      const int64_t v = words[i++];
      if (v < lo || v > hi) bad = true;
      return v;
    };
    auto raw = [&]() -> int64_t {
      if (bad || i >= n) {
        bad = true;
        return 0;
      }
      return words[i++];
    };
    if (next(kExportMagic, kExportMagic) != kExportMagic || next(kExportVersion, kExportVersion) != kExportVersion)
      return PA_ERR_INVALID;
    const int32_t nb = (int32_t)next(1, INT32_MAX), bs = (int32_t)next(1, INT32_MAX);
    const bool caching = next(0, 1) != 0;
    const int32_t ncpu = (int32_t)next(0, INT32_MAX);
    // every block takes at least three words below, and every swap block one
    // (in the swap pool's free queue or in a swapped-out table)
    if (bad || nb > n || ncpu > n) return PA_ERR_INVALID;
    std::unique_ptr<pa_alloc> a(new pa_alloc());
    a->num_blocks = nb;
    a->block_size = bs;
    a->caching = caching;
    a->cow_copies = next(0, INT64_MAX);
    a->alloc_failures = next(0, INT64_MAX);
    a->lookup_blocks = next(0, INT64_MAX);
    a->hit_blocks = next(0, INT64_MAX);
    a->evictions = next(0, INT64_MAX);
    a->ref.assign(nb, 0);
    a->prev.assign(nb, -1);
    a->next.assign(nb, -1);
    a->in_free.assign(nb, 0);
    a->hash.assign(nb, 0);
    a->has_hash.assign(nb, 0);
    const int64_t nfree = next(0, nb);
    for (int64_t k = 0; !bad && k < nfree; ++k) {
      const int32_t b = (int32_t)next(0, nb - 1);
      if (!bad && a->in_free[b]) bad = true;
      if (!bad) a->push_back(b);
    }
    for (int32_t b = 0; !bad && b < nb; ++b) a->ref[b] = (int32_t)next(0, INT32_MAX);
    for (int32_t b = 0; !bad && b < nb; ++b) a->has_hash[b] = (uint8_t)next(0, 1);
    for (int32_t b = 0; !bad && b < nb; ++b) a->hash[b] = (uint64_t)raw();
    for (int32_t b = 0; !bad && b < nb; ++b)
      if (a->in_free[b] && a->ref[b] != 0) bad = true;  // a free block has no owner
    const int64_t ncached = next(0, nb);
    for (int64_t k = 0; !bad && k < ncached; ++k) {
      const uint64_t h = (uint64_t)raw();
      const int32_t b = (int32_t)next(0, nb - 1);
      if (!bad && (!a->has_hash[b] || a->hash[b] != h || !a->cached.emplace(h, b).second)) bad = true;
    }
    const int64_t ncpu_free = next(0, ncpu);
    if (!bad && ncpu > 0) {
      a->num_cpu_blocks = ncpu;
      a->cpu.prev.assign(ncpu, -1);
      a->cpu.next.assign(ncpu, -1);
      std::vector<uint8_t> seen(ncpu, 0);
      for (int64_t k = 0; !bad && k < ncpu_free; ++k) {
        const int32_t b = (int32_t)next(0, ncpu - 1);
        if (bad || seen[b]) {
          bad = true;
          break;
        }
        seen[b] = 1;
        a->cpu.prev[b] = a->cpu.tail;  // append at the tail, in the exported order
        if (a->cpu.tail < 0) a->cpu.head = b; else a->cpu.next[a->cpu.tail] = b;
        a->cpu.tail = b;
        ++a->cpu.n;
      }
    }
    const int64_t nseq = next(0, n);
    for (int64_t k = 0; !bad && k < nseq; ++k) {
      const int id = (int)next(0, INT32_MAX);
      Seq q;
      q.num_tokens = next(0, INT64_MAX);
      q.salt = (uint64_t)raw();
      q.parent = (uint64_t)raw();
      q.hashable = next(0, 1) != 0;
      q.swapped = next(0, 1) != 0;
      if (q.swapped && ncpu == 0) bad = true;
      const int64_t nbk = next(0, n);
      const int32_t lim = q.swapped ? ncpu : nb;
      for (int64_t t = 0; !bad && t < nbk; ++t) q.blocks.push_back((int32_t)next(0, (int64_t)lim - 1));
      if (!bad && (int64_t)q.blocks.size() * bs < q.num_tokens) bad = true;  // tokens beyond the blocks
      const int64_t np = next(0, (int64_t)bs - 1);  // token ids of a block not yet full
      for (int64_t t = 0; !bad && t < np; ++t) q.pending.push_back((int32_t)next(INT32_MIN, INT32_MAX));
      if (!bad && !a->seqs.emplace(id, std::move(q)).second) bad = true;
    }
    if (!bad) {
      // refcounts are the number of resident tables holding the block, a
      // block is in the free queue exactly when nothing holds it, and every
      // swap block is either in the swap pool's free queue or held by exactly
      // one swapped-out table, exactly once (swap blocks are never shared)
      std::vector<int64_t> holders(nb, 0);
      std::vector<int64_t> cpu_holders(ncpu > 0 ? ncpu : 0, 0);
      std::vector<uint8_t> cpu_free(ncpu > 0 ? ncpu : 0, 0);
      for (int32_t b = a->cpu.head; ncpu > 0 && b >= 0; b = a->cpu.next[b]) cpu_free[b] = 1;
      for (const auto& kv : a->seqs)
        for (int32_t b : kv.second.blocks) {
          if (kv.second.swapped) {
            ++cpu_holders[b];
          } else {
            ++holders[b];
          }
        }
      for (int32_t b = 0; !bad && b < nb; ++b)
        if (holders[b] != a->ref[b] || (a->ref[b] == 0) != (a->in_free[b] != 0)) bad = true;
      for (int32_t b = 0; !bad && b < ncpu; ++b)
        if (cpu_holders[b] + cpu_free[b] != 1) bad = true;
      // every hashed block is the cache's entry for its hash
      int64_t hashed = 0;
      for (int32_t b = 0; b < nb; ++b) hashed += a->has_hash[b];
      if (hashed != (int64_t)a->cached.size()) bad = true;
    }
    if (bad || i != n) return PA_ERR_INVALID;
    *out = a.release();
    return PA_OK;
  });
}

}  // extern "C"
