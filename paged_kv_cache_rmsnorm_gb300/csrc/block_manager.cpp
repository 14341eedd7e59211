// Host-side block manager: the control plane that produces the block tables
// and slot mappings the attention step consumes.
//
// What the pages fix ("Nano-vLLM深度解读（下）" §4, the CPU-side Block Manager:
// it manages token sequences, allocates blocks, keeps reference counts and
// reuses cached prefixes; "同一个 Qwen3，两种写法" §3.3, the paged KV cache):
//   * the cache is one pool of fixed 256-token blocks allocated up front;
//   * each sequence owns a block table, logical block -> physical block;
//   * the slot of a token is physical block * 256 + offset in the block;
//   * blocks carry a reference count and a prefix hash, so sequences with the
//     same prefix point at the same physical blocks and store that KV once.
// Readings where the pages leave the policy open (the plainest ones):
//   * only full blocks are hashed; a block's hash chains the previous block's
//     hash with its 256 token ids (FNV-1a, 64 bit, over the bytes of the
//     previous hash and of the token ids); a lookup also compares the token
//     ids, so a hash collision never shares a block;
//   * at allocation the blocks of a prompt are matched from the first one on
//     and the first miss ends the reuse for the rest of the prompt (a later
//     block's hash covers the whole prefix anyway); reused blocks count as
//     cached tokens, which need no new KV;
//   * a freed block (reference count 0) keeps its contents and hash and goes
//     to the back of the free list, so it can still be reused by a later
//     prompt with the same prefix until the pool hands it out again;
//   * decode appends one token at a time: the token that starts a new block
//     takes a free block; the token that fills a block gives it its hash.
// One manager is not safe for concurrent use from several threads.
#include <cstdint>
#include <cstring>
#include <deque>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/pkv.h"

namespace pkv {
int report_error(int code, const char* fmt, ...);
}  // namespace pkv

namespace {

constexpr int kBlock = PKV_BLOCK_SIZE;
constexpr uint64_t kNoHash = ~uint64_t(0);

uint64_t fnv1a(uint64_t h, const void* data, size_t n) {
  const unsigned char* p = static_cast<const unsigned char*>(data);
  for (size_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= 1099511628211ull;  // FNV 64-bit prime
  }
  return h;
}

// Hash of a full block: FNV-1a over the little-endian bytes of the previous
// block's hash (all ones for the first block) and of the 256 token ids.
uint64_t block_hash(uint64_t prev, const int32_t* tokens) {
  uint64_t h = 14695981039346656037ull;  // FNV 64-bit offset basis
  unsigned char b[8];
  for (int i = 0; i < 8; ++i) b[i] = static_cast<unsigned char>(prev >> (8 * i));
  h = fnv1a(h, b, 8);
  for (int t = 0; t < kBlock; ++t) {
    const uint32_t v = static_cast<uint32_t>(tokens[t]);
    unsigned char c[4] = {static_cast<unsigned char>(v), static_cast<unsigned char>(v >> 8),
                          static_cast<unsigned char>(v >> 16), static_cast<unsigned char>(v >> 24)};
    h = fnv1a(h, c, 4);
  }
  return h == kNoHash ? h - 1 : h;  // kNoHash marks "no hash"
}

struct Block {
  int32_t ref = 0;
  uint64_t hash = kNoHash;
  std::vector<int32_t> tokens;  // the ids of a full, hashed block
};

struct Seq {
  std::vector<int32_t> tokens;
  std::vector<int32_t> table;  // logical block -> physical block
  int32_t num_cached = 0;      // leading tokens whose KV was already in reused blocks
};

}  // namespace

struct pkv_block_manager {
  std::vector<Block> blocks;
  std::deque<int32_t> free_list;
  std::unordered_map<uint64_t, int32_t> by_hash;
  std::unordered_map<int64_t, Seq> seqs;
  int64_t num_free = 0;

  int32_t take_free() {
    const int32_t b = free_list.front();
    free_list.pop_front();
    Block& blk = blocks[b];
    if (blk.hash != kNoHash) {  // its old contents are about to be overwritten
      auto it = by_hash.find(blk.hash);
      if (it != by_hash.end() && it->second == b) by_hash.erase(it);
    }
    blk.hash = kNoHash;
    blk.tokens.clear();
    blk.ref = 1;
    --num_free;
    return b;
  }

  void revive(int32_t b) {  // a freed block whose cached contents are reused
    for (auto it = free_list.begin(); it != free_list.end(); ++it)
      if (*it == b) {
        free_list.erase(it);
        break;
      }
    blocks[b].ref = 1;
    --num_free;
  }

  void set_hash(int32_t b, uint64_t h, const int32_t* tokens) {
    Block& blk = blocks[b];
    blk.hash = h;
    blk.tokens.assign(tokens, tokens + kBlock);
    by_hash[h] = b;
  }

  int32_t lookup(uint64_t h, const int32_t* tokens) const {
    auto it = by_hash.find(h);
    if (it == by_hash.end()) return -1;
    const Block& blk = blocks[it->second];
    if (blk.tokens.size() != static_cast<size_t>(kBlock) ||
        std::memcmp(blk.tokens.data(), tokens, kBlock * sizeof(int32_t)) != 0)
      return -1;
    return it->second;
  }
};

using pkv::report_error;

extern "C" {

pkv_block_manager* pkv_bm_create(int32_t num_blocks) {
  if (num_blocks <= 0) {
    report_error(PKV_ERR_SHAPE, "num_blocks must be > 0");
    return nullptr;
  }
  pkv_block_manager* bm = new (std::nothrow) pkv_block_manager();
  if (!bm) {
    report_error(PKV_ERR_SHAPE, "out of host memory");
    return nullptr;
  }
  bm->blocks.resize(num_blocks);
  for (int32_t b = 0; b < num_blocks; ++b) bm->free_list.push_back(b);
  bm->num_free = num_blocks;
  return bm;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

int64_t pkv_bm_num_free_blocks(const pkv_block_manager* bm) { return bm ? bm->num_free : -1; }

int32_t pkv_bm_ref_count(const pkv_block_manager* bm, int32_t block) {
  if (!bm || block < 0 || block >= static_cast<int32_t>(bm->blocks.size())) return -1;
  return bm->blocks[block].ref;
}

int pkv_bm_allocate(pkv_block_manager* bm, int64_t seq_id, const int32_t* token_ids, int32_t num_tokens,
                    int32_t* num_cached_tokens) {
  if (!bm || (!token_ids && num_tokens > 0)) return report_error(PKV_ERR_NULL, "a required pointer is NULL");
  if (num_tokens <= 0) return report_error(PKV_ERR_SHAPE, "a prompt needs at least one token");
  if (bm->seqs.count(seq_id)) return report_error(PKV_ERR_SHAPE, "sequence %lld is already allocated", (long long)seq_id);
  const int32_t need = (num_tokens + kBlock - 1) / kBlock;
  // worst case every block is new; checked up front so a failure changes nothing
  if (need > bm->num_free) return report_error(PKV_ERR_WORKSPACE, "%d blocks needed, %lld free", need, (long long)bm->num_free);
  Seq seq;
  seq.tokens.assign(token_ids, token_ids + num_tokens);
  uint64_t h = kNoHash;
  bool miss = false;
  for (int32_t i = 0; i < need; ++i) {
    const int32_t* tok = seq.tokens.data() + static_cast<size_t>(i) * kBlock;
    const bool full = (i + 1) * kBlock <= num_tokens;
    h = full ? block_hash(h, tok) : kNoHash;
    int32_t b = (!miss && full) ? bm->lookup(h, tok) : -1;
    if (b < 0) miss = true;
    if (miss) {
      b = bm->take_free();
    } else {
      seq.num_cached += kBlock;
      if (bm->blocks[b].ref > 0) ++bm->blocks[b].ref;
      else bm->revive(b);
    }
    if (full && bm->blocks[b].hash != h) bm->set_hash(b, h, tok);
    seq.table.push_back(b);
  }
  if (num_cached_tokens) *num_cached_tokens = seq.num_cached;
  bm->seqs.emplace(seq_id, std::move(seq));
  return PKV_OK;
}

int pkv_bm_append(pkv_block_manager* bm, int64_t seq_id, int32_t token_id, int32_t* slot) {
  if (!bm) return report_error(PKV_ERR_NULL, "a required pointer is NULL");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return report_error(PKV_ERR_SHAPE, "sequence %lld is not allocated", (long long)seq_id);
  Seq& seq = it->second;
  const int64_t len = static_cast<int64_t>(seq.tokens.size()) + 1;
  if (len % kBlock == 1) {  // the new token starts a block
    if (bm->num_free == 0) return report_error(PKV_ERR_WORKSPACE, "no free block");
    seq.table.push_back(bm->take_free());
  }
  seq.tokens.push_back(token_id);
  const int32_t last = seq.table.back();
  if (len % kBlock == 0) {  // the new token fills its block: the block gets its hash
    const size_t nb = seq.table.size();
    const uint64_t prev = nb >= 2 ? bm->blocks[seq.table[nb - 2]].hash : kNoHash;
    const int32_t* tok = seq.tokens.data() + (nb - 1) * kBlock;
    bm->set_hash(last, block_hash(prev, tok), tok);
  }
  if (slot) *slot = static_cast<int32_t>(static_cast<int64_t>(last) * kBlock + (len - 1) % kBlock);
  return PKV_OK;
}

int pkv_bm_free(pkv_block_manager* bm, int64_t seq_id) {
  if (!bm) return report_error(PKV_ERR_NULL, "a required pointer is NULL");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return report_error(PKV_ERR_SHAPE, "sequence %lld is not allocated", (long long)seq_id);
  const std::vector<int32_t>& table = it->second.table;
  for (auto b = table.rbegin(); b != table.rend(); ++b) {  // last blocks first: the prefix stays cached longest
    Block& blk = bm->blocks[*b];
    if (--blk.ref == 0) {
      bm->free_list.push_back(*b);
      ++bm->num_free;
    }
  }
  bm->seqs.erase(it);
  return PKV_OK;
}

int pkv_bm_seq_info(const pkv_block_manager* bm, int64_t seq_id, int32_t* num_tokens, int32_t* num_blocks,
                    int32_t* num_cached_tokens) {
  if (!bm) return report_error(PKV_ERR_NULL, "a required pointer is NULL");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return report_error(PKV_ERR_SHAPE, "sequence %lld is not allocated", (long long)seq_id);
  if (num_tokens) *num_tokens = static_cast<int32_t>(it->second.tokens.size());
  if (num_blocks) *num_blocks = static_cast<int32_t>(it->second.table.size());
  if (num_cached_tokens) *num_cached_tokens = it->second.num_cached;
  return PKV_OK;
}

int pkv_bm_block_table(const pkv_block_manager* bm, const int64_t* seq_ids, int32_t num_seqs, int32_t* table,
                       int32_t max_blocks) {
  if (!bm || (num_seqs > 0 && (!seq_ids || !table))) return report_error(PKV_ERR_NULL, "a required pointer is NULL");
  if (num_seqs < 0 || max_blocks <= 0) return report_error(PKV_ERR_SHAPE, "num_seqs < 0 or max_blocks <= 0");
  for (int32_t s = 0; s < num_seqs; ++s) {
    auto it = bm->seqs.find(seq_ids[s]);
    if (it == bm->seqs.end()) return report_error(PKV_ERR_SHAPE, "sequence %lld is not allocated", (long long)seq_ids[s]);
    const std::vector<int32_t>& t = it->second.table;
    if (static_cast<int32_t>(t.size()) > max_blocks)
      return report_error(PKV_ERR_SHAPE, "sequence %lld holds %zu blocks > max_blocks", (long long)seq_ids[s], t.size());
    int32_t* row = table + static_cast<int64_t>(s) * max_blocks;
    for (int32_t i = 0; i < max_blocks; ++i) row[i] = i < static_cast<int32_t>(t.size()) ? t[i] : -1;
  }
  return PKV_OK;
}

int pkv_bm_slot_mapping(const pkv_block_manager* bm, int64_t seq_id, int32_t start, int32_t end, int32_t* slots) {
  if (!bm || (end > start && !slots)) return report_error(PKV_ERR_NULL, "a required pointer is NULL");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return report_error(PKV_ERR_SHAPE, "sequence %lld is not allocated", (long long)seq_id);
  const std::vector<int32_t>& t = it->second.table;
  const int64_t len = static_cast<int64_t>(it->second.tokens.size());
  if (start < 0 || end < start || end > len) return report_error(PKV_ERR_SHAPE, "token range outside the sequence");
  for (int32_t p = start; p < end; ++p) slots[p - start] = t[p / kBlock] * kBlock + p % kBlock;
  return PKV_OK;
}

}  // extern "C"
