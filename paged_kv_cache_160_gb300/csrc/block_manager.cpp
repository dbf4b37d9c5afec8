// Host block manager: the free-block queue, per-block ref_cnt and per-sequence block
// tables of "PagedAttention: manage the KV cache like virtual memory" §3.2–§3.3, with
// fork and copy-on-write from "Lecture 33 — KV Cache management" §2.4 and preemption by
// swapping (a host-memory block pool with its own FIFO queue) from its §5.2, and prefix
// caching from "PagedAttention: manage the KV cache like virtual memory" §3.4–§3.5: a full
// block is named by a hash of its parent block's hash and its tokens; a hit re-uses the block
// (taking it out of the middle of the free queue if nobody held it), and a cached block that
// nobody holds stays reusable until it is popped for new data.
//
// The free queue is an intrusive doubly linked list over block ids (allocate pops the
// head, free pushes the tail, a claimed block is unlinked from the middle in O(1)).
// Every entry point validates first and mutates after, so a failing call leaves the
// manager unchanged.
#include <cstdint>
#include <deque>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pkv.h"

namespace {

struct Seq {
  std::vector<int32_t> blocks;   // device blocks, or host blocks while swapped out
  int64_t n_tokens = 0;
  bool swapped = false;
};

}  // namespace

struct pkv_block_manager {
  int num_blocks = 0;
  int block_size = 0;
  std::vector<int32_t> ref;
  std::vector<int32_t> prev, next;   // free-list links; -1 = none
  std::vector<uint8_t> in_free;
  int32_t head = -1, tail = -1;
  int num_free = 0;
  std::unordered_map<int64_t, Seq> seqs;
  std::vector<uint64_t> bhash;       // prefix-cache hash of a full block ...
  std::vector<uint8_t> has_hash;     // ... valid when set
  std::unordered_map<uint64_t, int32_t> hash_to_block;
  std::deque<int32_t> host_free;     // host swap pool: FIFO of free host block ids
  int num_host_blocks = 0;
  int num_swapped = 0;

  // A resident (not swapped out) sequence, or nullptr.
  Seq* resident(int64_t seq) {
    auto it = seqs.find(seq);
    return it == seqs.end() || it->second.swapped ? nullptr : &it->second;
  }

  void push_tail(int32_t b) {
    prev[b] = tail;
    next[b] = -1;
    if (tail >= 0) next[tail] = b; else head = b;
    tail = b;
    in_free[b] = 1;
    ++num_free;
  }
  void unlink(int32_t b) {
    if (prev[b] >= 0) next[prev[b]] = next[b]; else head = next[b];
    if (next[b] >= 0) prev[next[b]] = prev[b]; else tail = prev[b];
    prev[b] = next[b] = -1;
    in_free[b] = 0;
    --num_free;
  }
  int32_t pop_head() {  // caller checked num_free > 0
    int32_t b = head;
    unlink(b);
    ref[b] = 1;
    if (has_hash[b]) {    // the block gets new contents: its cached prefix is gone
      auto it = hash_to_block.find(bhash[b]);
      if (it != hash_to_block.end() && it->second == b) hash_to_block.erase(it);
      has_hash[b] = 0;
    }
    return b;
  }
  // Prefix-cache hit: one more holder; a block nobody held leaves the free queue.
  void touch(int32_t b) {
    if (in_free[b]) unlink(b);
    ++ref[b];
  }
  void release(int32_t b) {
    if (--ref[b] == 0) push_tail(b);
  }
  int64_t blocks_for(int64_t n_tokens) const { return (n_tokens + block_size - 1) / block_size; }

  // Blocks one append_slot on `s` would pop (0 or 1), given extra ref drops in `drop`.
  int pops_for_append(const Seq& s, int64_t n_tokens, const std::unordered_map<int32_t, int>* drop) const {
    if (n_tokens % block_size == 0) return 1;
    int32_t last = s.blocks[n_tokens / block_size];
    int r = ref[last];
    if (drop) {
      auto it = drop->find(last);
      if (it != drop->end()) r -= it->second;
    }
    return r > 1 ? 1 : 0;
  }

  // Appends one token; the caller guaranteed a free block when one is needed.
  int64_t append(Seq& s, int32_t* cow_src, int32_t* cow_dst) {
    const int64_t p = s.n_tokens;
    *cow_src = -1;
    *cow_dst = -1;
    if (p % block_size == 0) {
      s.blocks.push_back(pop_head());
    } else {
      int32_t& last = s.blocks[p / block_size];
      if (ref[last] > 1) {
        int32_t fresh = pop_head();
        --ref[last];
        *cow_src = last;
        *cow_dst = fresh;
        last = fresh;
      }
    }
    s.n_tokens = p + 1;
    return int64_t(s.blocks[p / block_size]) * block_size + p % block_size;
  }
};

extern "C" {

pkv_status pkv_bm_create(int num_blocks, int block_size, pkv_block_manager** out) {
  if (!out || num_blocks <= 0 || block_size <= 0) return PKV_ERR_INVALID_ARG;
  auto* bm = new (std::nothrow) pkv_block_manager();
  if (!bm) return PKV_ERR_INVALID_ARG;
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->ref.assign(num_blocks, 0);
  bm->prev.assign(num_blocks, -1);
  bm->next.assign(num_blocks, -1);
  bm->in_free.assign(num_blocks, 0);
  bm->bhash.assign(num_blocks, 0);
  bm->has_hash.assign(num_blocks, 0);
  for (int b = 0; b < num_blocks; ++b) bm->push_tail(b);
  *out = bm;
  return PKV_OK;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

pkv_status pkv_bm_import_seq(pkv_block_manager* bm, int64_t seq, const int32_t* blocks, int n_blocks,
                             int n_tokens) {
  if (!bm || n_tokens < 0 || n_blocks < 0 || (n_blocks > 0 && !blocks)) return PKV_ERR_INVALID_ARG;
  if (bm->seqs.count(seq)) return PKV_ERR_INVALID_ARG;
  if (bm->blocks_for(n_tokens) != n_blocks) return PKV_ERR_INVALID_ARG;
  for (int i = 0; i < n_blocks; ++i)
    if (blocks[i] < 0 || blocks[i] >= bm->num_blocks) return PKV_ERR_INVALID_ARG;
  Seq s;
  s.blocks.assign(blocks, blocks + n_blocks);
  s.n_tokens = n_tokens;
  for (int32_t b : s.blocks) {
    if (bm->in_free[b]) bm->unlink(b);
    ++bm->ref[b];
  }
  bm->seqs.emplace(seq, std::move(s));
  return PKV_OK;
}

pkv_status pkv_bm_allocate(pkv_block_manager* bm, int64_t seq, int n_tokens) {
  if (!bm || n_tokens < 0 || bm->seqs.count(seq)) return PKV_ERR_INVALID_ARG;
  int64_t need = bm->blocks_for(n_tokens);
  if (need > bm->num_free) return PKV_ERR_NO_BLOCKS;
  Seq s;
  s.n_tokens = n_tokens;
  for (int64_t i = 0; i < need; ++i) s.blocks.push_back(bm->pop_head());
  bm->seqs.emplace(seq, std::move(s));
  return PKV_OK;
}

pkv_status pkv_bm_append_slot(pkv_block_manager* bm, int64_t seq, int64_t* slot, int32_t* cow_src,
                              int32_t* cow_dst) {
  if (!bm || !slot || !cow_src || !cow_dst) return PKV_ERR_INVALID_ARG;
  Seq* sq = bm->resident(seq);
  if (!sq) return PKV_ERR_INVALID_ARG;
  if (bm->pops_for_append(*sq, sq->n_tokens, nullptr) > bm->num_free) return PKV_ERR_NO_BLOCKS;
  *slot = bm->append(*sq, cow_src, cow_dst);
  return PKV_OK;
}

pkv_status pkv_bm_append_slots(pkv_block_manager* bm, int64_t seq, int n, int64_t* slots, int32_t* cow_pairs,
                               int* n_cow) {
  if (!bm || n < 0 || (n > 0 && (!slots || !cow_pairs)) || !n_cow) return PKV_ERR_INVALID_ARG;
  Seq* sq = bm->resident(seq);
  if (!sq) return PKV_ERR_INVALID_ARG;
  Seq& s = *sq;
  // Pops needed: a copy-on-write of the current last block (if shared and partially
  // filled) plus one block per block boundary crossed.
  int64_t need = 0;
  if (n > 0) {
    need += bm->pops_for_append(s, s.n_tokens, nullptr) && (s.n_tokens % bm->block_size != 0) ? 1 : 0;
    int64_t first_new = bm->blocks_for(s.n_tokens);
    int64_t last_needed = bm->blocks_for(s.n_tokens + n);
    need += last_needed - first_new;
  }
  if (need > bm->num_free) return PKV_ERR_NO_BLOCKS;
  int nc = 0;
  for (int i = 0; i < n; ++i) {
    int32_t cs, cd;
    slots[i] = bm->append(s, &cs, &cd);
    if (cs >= 0) {
      cow_pairs[2 * nc] = cs;
      cow_pairs[2 * nc + 1] = cd;
      ++nc;
    }
  }
  *n_cow = nc;
  return PKV_OK;
}

pkv_status pkv_bm_step_decode(pkv_block_manager* bm, const int64_t* seqs, int n, int max_blocks,
                              int64_t* slot_mapping, int32_t* cow_pairs, int* n_cow, int32_t* tables,
                              int32_t* lens) {
  if (!bm || n < 0 || max_blocks < 0 || !n_cow) return PKV_ERR_INVALID_ARG;
  if (n > 0 && (!seqs || !slot_mapping || !cow_pairs || !tables || !lens)) return PKV_ERR_INVALID_ARG;
  // Validate and count pops before changing anything.  A shared block copied by one
  // sequence of the batch may no longer be shared when a later sequence reaches it.
  std::unordered_set<int64_t> seen;
  std::unordered_map<int32_t, int> drop;
  int64_t need = 0;
  for (int i = 0; i < n; ++i) {
    const Seq* sq = bm->resident(seqs[i]);
    if (!sq || !seen.insert(seqs[i]).second) return PKV_ERR_INVALID_ARG;
    const Seq& s = *sq;
    if (bm->blocks_for(s.n_tokens + 1) > max_blocks) return PKV_ERR_INVALID_ARG;
    int pops = bm->pops_for_append(s, s.n_tokens, &drop);
    if (pops && s.n_tokens % bm->block_size != 0) ++drop[s.blocks[s.n_tokens / bm->block_size]];
    need += pops;
  }
  if (need > bm->num_free) return PKV_ERR_NO_BLOCKS;
  int nc = 0;
  for (int i = 0; i < n; ++i) {
    Seq& s = bm->seqs[seqs[i]];
    int32_t cs, cd;
    slot_mapping[i] = bm->append(s, &cs, &cd);
    if (cs >= 0) {
      cow_pairs[2 * nc] = cs;
      cow_pairs[2 * nc + 1] = cd;
      ++nc;
    }
  }
  *n_cow = nc;
  return pkv_bm_export(bm, seqs, n, max_blocks, tables, lens);
}

pkv_status pkv_bm_fork(pkv_block_manager* bm, int64_t parent, int64_t child) {
  if (!bm) return PKV_ERR_INVALID_ARG;
  const Seq* ps = bm->resident(parent);
  if (!ps || bm->seqs.count(child)) return PKV_ERR_INVALID_ARG;
  Seq c = *ps;
  for (int32_t b : c.blocks) ++bm->ref[b];
  bm->seqs.emplace(child, std::move(c));
  return PKV_OK;
}

pkv_status pkv_bm_free(pkv_block_manager* bm, int64_t seq) {
  if (!bm) return PKV_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
  if (it->second.swapped) {                  // its host blocks go back to the host queue
    for (int32_t b : it->second.blocks) bm->host_free.push_back(b);
    --bm->num_swapped;
  } else {
    for (int32_t b : it->second.blocks) bm->release(b);
  }
  bm->seqs.erase(it);
  return PKV_OK;
}

pkv_status pkv_bm_export(const pkv_block_manager* bm, const int64_t* seqs, int n, int max_blocks,
                         int32_t* tables, int32_t* lens) {
  if (!bm || n < 0 || max_blocks < 0) return PKV_ERR_INVALID_ARG;
  if (n > 0 && (!seqs || !tables || !lens)) return PKV_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seqs[i]);
    if (it == bm->seqs.end() || it->second.swapped || int64_t(it->second.blocks.size()) > max_blocks)
      return PKV_ERR_INVALID_ARG;
    if (it->second.n_tokens > INT32_MAX) return PKV_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n; ++i) {
    const Seq& s = bm->seqs.at(seqs[i]);
    int32_t* row = tables + int64_t(i) * max_blocks;
    size_t k = 0;
    for (; k < s.blocks.size(); ++k) row[k] = s.blocks[k];
    for (; k < size_t(max_blocks); ++k) row[k] = -1;
    lens[i] = int32_t(s.n_tokens);
  }
  return PKV_OK;
}

// 64-bit FNV-1a over the parent hash (8 bytes, little-endian) then the block's token ids
// (4 bytes each, little-endian); the first block's parent hash is the FNV offset basis.
static uint64_t fnv1a_block(uint64_t parent, const int32_t* tokens, int n) {
  uint64_t h = 0xcbf29ce484222325ull;
  auto mix = [&](uint8_t byte) {
    h ^= byte;
    h *= 0x100000001b3ull;
  };
  for (int i = 0; i < 8; ++i) mix(uint8_t(parent >> (8 * i)));
  for (int t = 0; t < n; ++t) {
    const uint32_t u = uint32_t(tokens[t]);
    for (int i = 0; i < 4; ++i) mix(uint8_t(u >> (8 * i)));
  }
  return h;
}

pkv_status pkv_bm_allocate_cached(pkv_block_manager* bm, int64_t seq, const int32_t* tokens, int n_tokens,
                                  int* n_cached_tokens) {
  if (!bm || n_tokens < 0 || (n_tokens > 0 && !tokens) || !n_cached_tokens || bm->seqs.count(seq))
    return PKV_ERR_INVALID_ARG;
  const int bs = bm->block_size;
  const int n_full = n_tokens / bs;
  const int64_t need_total = bm->blocks_for(n_tokens);
  // Longest run of cached full blocks from the start (the hash chain makes it a prefix).
  std::vector<uint64_t> hashes(n_full);
  std::vector<int32_t> hits;
  uint64_t parent = 0xcbf29ce484222325ull;
  int held_free = 0;                         // hits now in the free queue (they leave it)
  for (int i = 0; i < n_full; ++i) {
    hashes[i] = fnv1a_block(parent, tokens + int64_t(i) * bs, bs);
    parent = hashes[i];
    if (int(hits.size()) == i) {
      auto it = bm->hash_to_block.find(hashes[i]);
      if (it != bm->hash_to_block.end()) {
        hits.push_back(it->second);
        if (bm->ref[it->second] == 0) ++held_free;
      }
    }
  }
  const int64_t misses = need_total - int64_t(hits.size());
  if (misses > bm->num_free - held_free) return PKV_ERR_NO_BLOCKS;
  Seq s;
  s.n_tokens = n_tokens;
  for (int32_t b : hits) {
    bm->touch(b);
    s.blocks.push_back(b);
  }
  for (int64_t i = int64_t(hits.size()); i < need_total; ++i) {
    const int32_t b = bm->pop_head();
    s.blocks.push_back(b);
    if (i < n_full && !bm->hash_to_block.count(hashes[i])) {   // register the new full block
      bm->bhash[b] = hashes[i];
      bm->has_hash[b] = 1;
      bm->hash_to_block.emplace(hashes[i], b);
    }
  }
  *n_cached_tokens = int(hits.size()) * bs;
  bm->seqs.emplace(seq, std::move(s));
  return PKV_OK;
}

int pkv_bm_block_hash(const pkv_block_manager* bm, int block, uint64_t* hash) {
  if (!bm || block < 0 || block >= bm->num_blocks || !hash) return -1;
  if (!bm->has_hash[block]) return 0;
  *hash = bm->bhash[block];
  return 1;
}

int pkv_bm_num_cached(const pkv_block_manager* bm) { return bm ? int(bm->hash_to_block.size()) : -1; }

pkv_status pkv_bm_set_host_pool(pkv_block_manager* bm, int num_host_blocks) {
  if (!bm || num_host_blocks < 0 || bm->num_swapped > 0) return PKV_ERR_INVALID_ARG;
  bm->num_host_blocks = num_host_blocks;
  bm->host_free.clear();
  for (int b = 0; b < num_host_blocks; ++b) bm->host_free.push_back(b);
  return PKV_OK;
}

pkv_status pkv_bm_swap_out(pkv_block_manager* bm, int64_t seq, int32_t* pairs, int max_pairs, int* n_pairs) {
  if (!bm || !n_pairs || max_pairs < 0) return PKV_ERR_INVALID_ARG;
  Seq* sq = bm->resident(seq);
  if (!sq || int64_t(sq->blocks.size()) > max_pairs || (!sq->blocks.empty() && !pairs)) return PKV_ERR_INVALID_ARG;
  if (sq->blocks.size() > bm->host_free.size()) return PKV_ERR_NO_BLOCKS;
  // Each table entry gets a host block (in table order); then the device blocks are released
  // in table order, as if the sequence were freed.  A block shared with another sequence
  // stays on the device for it; this sequence takes its own host copy.
  std::vector<int32_t> host(sq->blocks.size());
  for (size_t i = 0; i < sq->blocks.size(); ++i) {
    host[i] = bm->host_free.front();
    bm->host_free.pop_front();
    pairs[2 * i] = sq->blocks[i];
    pairs[2 * i + 1] = host[i];
  }
  for (int32_t b : sq->blocks) bm->release(b);
  sq->blocks = std::move(host);
  sq->swapped = true;
  ++bm->num_swapped;
  *n_pairs = int(sq->blocks.size());
  return PKV_OK;
}

pkv_status pkv_bm_swap_in(pkv_block_manager* bm, int64_t seq, int32_t* pairs, int max_pairs, int* n_pairs) {
  if (!bm || !n_pairs || max_pairs < 0) return PKV_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end() || !it->second.swapped) return PKV_ERR_INVALID_ARG;
  Seq& s = it->second;
  if (int64_t(s.blocks.size()) > max_pairs || (!s.blocks.empty() && !pairs)) return PKV_ERR_INVALID_ARG;
  if (int64_t(s.blocks.size()) > bm->num_free) return PKV_ERR_NO_BLOCKS;
  // Each host block gets a fresh device block (popped in table order); the host blocks
  // return to the tail of the host queue in table order.
  std::vector<int32_t> dev(s.blocks.size());
  for (size_t i = 0; i < s.blocks.size(); ++i) {
    dev[i] = bm->pop_head();
    pairs[2 * i] = s.blocks[i];
    pairs[2 * i + 1] = dev[i];
  }
  for (int32_t b : s.blocks) bm->host_free.push_back(b);
  s.blocks = std::move(dev);
  s.swapped = false;
  --bm->num_swapped;
  *n_pairs = int(s.blocks.size());
  return PKV_OK;
}

int pkv_bm_num_free_host(const pkv_block_manager* bm) { return bm ? int(bm->host_free.size()) : -1; }

int pkv_bm_is_swapped(const pkv_block_manager* bm, int64_t seq) {
  if (!bm) return -1;
  auto it = bm->seqs.find(seq);
  return it == bm->seqs.end() ? -1 : (it->second.swapped ? 1 : 0);
}

int pkv_bm_ref_cnt(const pkv_block_manager* bm, int block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return -1;
  return bm->ref[block];
}

int pkv_bm_num_free(const pkv_block_manager* bm) { return bm ? bm->num_free : -1; }

int pkv_bm_free_queue(const pkv_block_manager* bm, int32_t* out, int max_n) {
  if (!bm) return -1;
  int k = 0;
  for (int32_t b = bm->head; b >= 0; b = bm->next[b]) {
    if (out && k < max_n) out[k] = b;
    ++k;
  }
  return k;
}

}  // extern "C"
