// Request-level KV cache allocator.
//
// "KV Cache 管理设计文档" (cann-recipes-infer): §2.2 KVCacheManager (allocate_slots,
// get_block_ids, free, format_usage), §2.3 SingleTypeKVCacheManager
// (get_num_blocks_to_allocate, allocate_new_blocks, remove_skipped_blocks, free,
// get_num_skipped_tokens), §2.3.2 the null-padded sliding-window layout, §2.4
// BlockPool, §3.3 the two-phase allocate_slots, §4.2.2 prepare_block_tables.
// "KV Cache 笔记" (HF continuous batching): block fingerprints chained from the
// parent block, the tokens and the layer group, prefix match, and fork_blocks
// (full blocks shared by reference count, the incomplete last block copied), with a
// process-independent hash (BLAKE2b, 8-byte digest).
//
// Readings where the pages leave a step open:
//  * The leading null entries of a sliding-window list are the blocks wholly before
//    position computed - W + 1, the first key a query of this step can see; the
//    paged prefill reads the cache through the table, so every visible position
//    keeps a real block.
//  * Released blocks go back to the queue tail in the request's logical order.
//  * A fingerprint is forgotten when its block's last reference is released.
//  * Prefix matching covers full blocks only, never the block of the last token.
//  * One manager per attention type, each with its own pool; group id = type index.
#include <cstring>
#include <string>
#include <unordered_map>
#include <vector>

#include "abi_common.h"
#include "host_pool.h"

namespace pkv {
namespace {

// ------------------------------------------------------------------ BLAKE2b
// RFC 7693: 12 rounds of the G mixing function over a 16-word state; the
// initial chaining value is the SHA-512 IV with the parameter block (digest
// length, key length 0, fanout 1, depth 1) folded into word 0.
constexpr uint64_t kIV[8] = {
    0x6a09e667f3bcc908ULL, 0xbb67ae8584caa73bULL, 0x3c6ef372fe94f82bULL, 0xa54ff53a5f1d36f1ULL,
    0x510e527fade682d1ULL, 0x9b05688c2b3e6c1fULL, 0x1f83d9abfb41bd6bULL, 0x5be0cd19137e2179ULL};

constexpr uint8_t kSigma[12][16] = {
    {0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15},
    {14, 10, 4, 8, 9, 15, 13, 6, 1, 12, 0, 2, 11, 7, 5, 3},
    {11, 8, 12, 0, 5, 2, 15, 13, 10, 14, 3, 6, 7, 1, 9, 4},
    {7, 9, 3, 1, 13, 12, 11, 14, 2, 6, 5, 10, 4, 0, 15, 8},
    {9, 0, 5, 7, 2, 4, 10, 15, 14, 1, 11, 12, 6, 8, 3, 13},
    {2, 12, 6, 10, 0, 11, 8, 3, 4, 13, 7, 5, 15, 14, 1, 9},
    {12, 5, 1, 15, 14, 13, 4, 10, 0, 7, 6, 3, 9, 2, 8, 11},
    {13, 11, 7, 14, 12, 1, 3, 9, 5, 0, 15, 4, 8, 6, 2, 10},
    {6, 15, 14, 9, 11, 3, 0, 8, 12, 2, 13, 7, 1, 4, 10, 5},
    {10, 2, 8, 4, 7, 6, 1, 5, 15, 11, 9, 14, 3, 12, 13, 0},
    {0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15},
    {14, 10, 4, 8, 9, 15, 13, 6, 1, 12, 0, 2, 11, 7, 5, 3}};

inline uint64_t rotr64(uint64_t x, int n) { return (x >> n) | (x << (64 - n)); }

inline uint64_t load_le64(const uint8_t* p) {
  uint64_t v = 0;
  for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];
  return v;
}

class Blake2b {
 public:
  explicit Blake2b(int digest_bytes) : outlen_(digest_bytes) {
    for (int i = 0; i < 8; ++i) h_[i] = kIV[i];
    h_[0] ^= 0x01010000ULL ^ (uint64_t)digest_bytes;  // no key
  }
  void update(const uint8_t* data, size_t n) {
    for (size_t i = 0; i < n; ++i) {
      if (fill_ == 128) {  // a full buffer is compressed only once more input follows
        t_ += 128;
        compress(false);
        fill_ = 0;
      }
      buf_[fill_++] = data[i];
    }
  }
  // Digest bytes, little-endian words; returns the first 8 as a little-endian u64.
  uint64_t final64() {
    t_ += fill_;
    while (fill_ < 128) buf_[fill_++] = 0;
    compress(true);
    uint64_t out = 0;
    for (int i = outlen_ - 1; i >= 0; --i) out = (out << 8) | (uint8_t)(h_[i / 8] >> (8 * (i % 8)));
    return out;
  }

 private:
  void compress(bool last) {
    uint64_t m[16], v[16];
    for (int i = 0; i < 16; ++i) m[i] = load_le64(buf_ + 8 * i);
    for (int i = 0; i < 8; ++i) {
      v[i] = h_[i];
      v[i + 8] = kIV[i];
    }
    v[12] ^= t_;  // low word of the byte counter (inputs here stay far below 2^64)
    if (last) v[14] = ~v[14];
    auto g = [&](int a, int b, int c, int d, uint64_t x, uint64_t y) {
      v[a] = v[a] + v[b] + x;
      v[d] = rotr64(v[d] ^ v[a], 32);
      v[c] = v[c] + v[d];
      v[b] = rotr64(v[b] ^ v[c], 24);
      v[a] = v[a] + v[b] + y;
      v[d] = rotr64(v[d] ^ v[a], 16);
      v[c] = v[c] + v[d];
      v[b] = rotr64(v[b] ^ v[c], 63);
    };
    for (int r = 0; r < 12; ++r) {
      const uint8_t* s = kSigma[r];
      g(0, 4, 8, 12, m[s[0]], m[s[1]]);
      g(1, 5, 9, 13, m[s[2]], m[s[3]]);
      g(2, 6, 10, 14, m[s[4]], m[s[5]]);
      g(3, 7, 11, 15, m[s[6]], m[s[7]]);
      g(0, 5, 10, 15, m[s[8]], m[s[9]]);
      g(1, 6, 11, 12, m[s[10]], m[s[11]]);
      g(2, 7, 8, 13, m[s[12]], m[s[13]]);
      g(3, 4, 9, 14, m[s[14]], m[s[15]]);
    }
    for (int i = 0; i < 8; ++i) h_[i] ^= v[i] ^ v[i + 8];
  }

  uint64_t h_[8];
  uint8_t buf_[128] = {};
  size_t fill_ = 0;
  uint64_t t_ = 0;
  int outlen_;
};

void put_le(std::vector<uint8_t>& b, uint64_t v, int bytes) {
  for (int i = 0; i < bytes; ++i) b.push_back((uint8_t)(v >> (8 * i)));
}

uint64_t block_hash(uint64_t parent, bool has_parent, const int32_t* tokens, int64_t n,
                    int32_t group_id) {
  std::vector<uint8_t> bytes;
  bytes.reserve(8 + 4 * n + 4);
  if (has_parent) put_le(bytes, parent, 8);
  for (int64_t i = 0; i < n; ++i) put_le(bytes, (uint32_t)tokens[i], 4);
  put_le(bytes, (uint32_t)group_id, 4);
  Blake2b h(8);
  h.update(bytes.data(), bytes.size());
  return h.final64();
}

}  // namespace
}  // namespace pkv

namespace pkv {
namespace {

// One attention type: its pool and the logical block lists of the requests.
struct TypeManager {
  pkv_pool pool;
  int32_t block_size = 0;
  int32_t window = 0;  // 0 = full attention
  int32_t group_id = 0;
  bool prefix = false;
  std::unordered_map<int64_t, std::vector<int32_t>> req_blocks;
  std::unordered_map<int64_t, std::vector<uint64_t>> req_hashes;
  std::unordered_map<uint64_t, int32_t> hash_to_block;
  std::unordered_map<int32_t, uint64_t> block_to_hash;

  int32_t null() const { return pool.null_block; }

  int64_t skipped_tokens(int64_t computed) const {
    if (window <= 0) return 0;
    const int64_t s = computed - window + 1;
    return s > 0 ? s : 0;
  }

  void release(const std::vector<int32_t>& ids) {
    std::vector<int32_t> freed;
    pool_release(&pool, ids.data(), (int64_t)ids.size(), &freed);
    for (int32_t b : freed) {
      auto it = block_to_hash.find(b);
      if (it != block_to_hash.end()) {
        hash_to_block.erase(it->second);
        block_to_hash.erase(it);
      }
    }
  }

  // remove_skipped_blocks: entries wholly before the first visible position become
  // the null block and their blocks are released.
  void remove_skipped(int64_t req, int64_t computed) {
    auto it = req_blocks.find(req);
    if (it == req_blocks.end()) return;
    std::vector<int32_t>& row = it->second;
    const int64_t n_skip = skipped_tokens(computed) / block_size;
    std::vector<int32_t> freed;
    for (int64_t j = 0; j < n_skip && j < (int64_t)row.size(); ++j) {
      if (row[j] != null()) {
        freed.push_back(row[j]);
        row[j] = null();
      }
    }
    release(freed);
  }

  // (logical entries, leading null entries) of a list covering num_tokens.
  void layout(int64_t num_tokens, int64_t computed, int64_t* nblk, int64_t* n_null) const {
    *nblk = ceil_div(num_tokens, block_size);
    const int64_t nn = skipped_tokens(computed) / block_size;
    *n_null = nn < *nblk ? nn : *nblk;
  }

  int64_t held(int64_t req) const {
    auto it = req_blocks.find(req);
    return it == req_blocks.end() ? 0 : (int64_t)it->second.size();
  }

  int64_t blocks_to_allocate(int64_t req, int64_t num_tokens, int64_t computed) const {
    int64_t nblk, n_null;
    layout(num_tokens, computed, &nblk, &n_null);
    int64_t n = 0;
    for (int64_t j = held(req); j < nblk; ++j) n += (j >= n_null);
    return n;
  }

  void allocate(int64_t req, int64_t num_tokens, int64_t computed) {
    int64_t nblk, n_null;
    layout(num_tokens, computed, &nblk, &n_null);
    const int64_t n_new = blocks_to_allocate(req, num_tokens, computed);
    std::vector<int32_t> fresh(n_new);
    pool_take(&pool, n_new, fresh.data());
    std::vector<int32_t>& row = req_blocks[req];
    int64_t k = 0;
    for (int64_t j = (int64_t)row.size(); j < nblk; ++j) row.push_back(j < n_null ? null() : fresh[k++]);
  }

  void free_request(int64_t req) {
    auto it = req_blocks.find(req);
    if (it == req_blocks.end()) return;
    std::vector<int32_t> ids;
    for (int32_t b : it->second)
      if (b != null()) ids.push_back(b);
    req_blocks.erase(it);
    req_hashes.erase(req);
    release(ids);
  }

  // Fingerprint chain of the leading full blocks of tokens, up to max_blocks.
  std::vector<uint64_t> chain(const int32_t* tokens, int64_t n_blocks) const {
    std::vector<uint64_t> h;
    h.reserve(n_blocks);
    for (int64_t j = 0; j < n_blocks; ++j)
      h.push_back(block_hash(j ? h[j - 1] : 0, j > 0, tokens + j * block_size, block_size, group_id));
    return h;
  }

  void cache_full_blocks(int64_t req, const int32_t* tokens, int64_t num_tokens) {
    if (!prefix) return;
    auto it = req_blocks.find(req);
    if (it == req_blocks.end()) return;
    const std::vector<int32_t>& row = it->second;
    std::vector<uint64_t>& hashes = req_hashes[req];
    int64_t n_full = num_tokens / block_size;
    if (n_full > (int64_t)row.size()) n_full = (int64_t)row.size();
    for (int64_t j = (int64_t)hashes.size(); j < n_full; ++j) {
      const uint64_t h = block_hash(j ? hashes[j - 1] : 0, j > 0, tokens + j * block_size,
                                    block_size, group_id);
      hashes.push_back(h);
      const int32_t b = row[j];
      if (b != null() && !hash_to_block.count(h) && !block_to_hash.count(b)) {
        hash_to_block[h] = b;
        block_to_hash[b] = h;
      }
    }
  }

  // Blocks of the longest fingerprinted prefix (never the block of the last token).
  std::vector<int32_t> match(const int32_t* tokens, int64_t num_tokens) const {
    std::vector<int32_t> out;
    if (!prefix || num_tokens < 1) return out;
    const int64_t limit = (num_tokens - 1) / block_size;
    uint64_t parent = 0;
    for (int64_t j = 0; j < limit; ++j) {
      const uint64_t h = block_hash(parent, j > 0, tokens + j * block_size, block_size, group_id);
      auto it = hash_to_block.find(h);
      if (it == hash_to_block.end()) break;
      out.push_back(it->second);
      parent = h;
    }
    return out;
  }
};

}  // namespace
}  // namespace pkv

struct pkv_kv_manager {
  std::vector<pkv::TypeManager> types;
  int32_t block_size = 0;
  int64_t max_model_len = 0;
};

extern "C" {

int pkv_manager_create(int32_t num_types, const int32_t* windows, const int64_t* num_blocks,
                       const int32_t* const* initial_orders, int32_t block_size,
                       int64_t max_model_len, int32_t prefix_caching, pkv_kv_manager** out) {
  PKV_REQUIRE(out && windows && num_blocks && num_types >= 1 && num_types <= 2 && block_size > 0 &&
                  max_model_len > 0,
              PKV_ERR_INVALID_ARG, "pkv_manager_create: bad args");
  PKV_REQUIRE(num_types == 1 || ((windows[0] > 0) != (windows[1] > 0)), PKV_ERR_INVALID_ARG,
              "pkv_manager_create: one manager per attention type (one full, one sliding)");
  auto* m = new pkv_kv_manager();
  m->block_size = block_size;
  m->max_model_len = max_model_len;
  m->types.resize(num_types);
  for (int32_t i = 0; i < num_types; ++i) {
    pkv_pool* p = nullptr;
    const int32_t* order = initial_orders ? initial_orders[i] : nullptr;
    const int rc = windows[i] < 0 ? PKV_ERR_INVALID_ARG : pkv_pool_create(num_blocks[i], order, &p);
    if (rc != PKV_OK) {
      delete m;
      if (windows[i] < 0) PKV_FAIL(PKV_ERR_INVALID_ARG, "pkv_manager_create: negative window");
      return rc;
    }
    pkv::TypeManager& t = m->types[i];
    t.pool = std::move(*p);
    pkv_pool_destroy(p);
    t.block_size = block_size;
    t.window = windows[i];
    t.group_id = i;
    t.prefix = prefix_caching != 0 && windows[i] == 0;
  }
  *out = m;
  pkv::clear_error();
  return PKV_OK;
}

void pkv_manager_destroy(pkv_kv_manager* mgr) { delete mgr; }

int pkv_manager_allocate_slots(pkv_kv_manager* mgr, int64_t request_id, int64_t computed_tokens,
                               int64_t num_new_tokens, int64_t lookahead_tokens) {
  PKV_REQUIRE(mgr && computed_tokens >= 0 && num_new_tokens >= 0 && lookahead_tokens >= 0,
              PKV_ERR_INVALID_ARG, "pkv_manager_allocate_slots: bad args");
  const int64_t total_computed =
      computed_tokens < mgr->max_model_len ? computed_tokens : mgr->max_model_len;
  int64_t need = computed_tokens + num_new_tokens + lookahead_tokens;
  if (need > mgr->max_model_len) need = mgr->max_model_len;
  // Phase 1: recycle, count, check (stop at the first type that cannot supply).
  for (pkv::TypeManager& t : mgr->types) {
    t.remove_skipped(request_id, total_computed);
    if ((int64_t)t.pool.queue.size() < t.blocks_to_allocate(request_id, need, total_computed))
      return 0;
  }
  // Phase 2: every type can supply its blocks.
  for (pkv::TypeManager& t : mgr->types) t.allocate(request_id, need, total_computed);
  return 1;
}

int64_t pkv_manager_get_block_ids(const pkv_kv_manager* mgr, int64_t request_id, int32_t type,
                                  int32_t* ids_out, int64_t capacity) {
  PKV_REQUIRE(mgr && type >= 0 && type < (int32_t)mgr->types.size() && capacity >= 0 &&
                  (ids_out || capacity == 0),
              PKV_ERR_INVALID_ARG, "pkv_manager_get_block_ids: bad args");
  const auto& rb = mgr->types[type].req_blocks;
  auto it = rb.find(request_id);
  if (it == rb.end()) return 0;
  const int64_t n = (int64_t)it->second.size();
  for (int64_t i = 0; i < n && i < capacity; ++i) ids_out[i] = it->second[i];
  return n;
}

int pkv_manager_free(pkv_kv_manager* mgr, int64_t request_id) {
  PKV_REQUIRE(mgr, PKV_ERR_INVALID_ARG, "pkv_manager_free: NULL manager");
  for (pkv::TypeManager& t : mgr->types) t.free_request(request_id);
  return PKV_OK;
}

int64_t pkv_manager_num_free(const pkv_kv_manager* mgr, int32_t type) {
  if (!mgr || type < 0 || type >= (int32_t)mgr->types.size()) return -1;
  return (int64_t)mgr->types[type].pool.queue.size();
}

int32_t pkv_manager_null_block(const pkv_kv_manager* mgr, int32_t type) {
  if (!mgr || type < 0 || type >= (int32_t)mgr->types.size()) return -1;
  return mgr->types[type].null();
}

int32_t pkv_manager_ref_count(const pkv_kv_manager* mgr, int32_t type, int32_t block) {
  if (!mgr || type < 0 || type >= (int32_t)mgr->types.size()) return -1;
  return pkv_pool_ref_count(&mgr->types[type].pool, block);
}

int64_t pkv_manager_format_usage(const pkv_kv_manager* mgr, char* buf, int64_t capacity) {
  PKV_REQUIRE(mgr && capacity >= 0 && (buf || capacity == 0), PKV_ERR_INVALID_ARG,
              "pkv_manager_format_usage: bad args");
  std::string s;
  for (size_t i = 0; i < mgr->types.size(); ++i) {
    const pkv::TypeManager& t = mgr->types[i];
    const int64_t used = t.pool.num_blocks - 1 - (int64_t)t.pool.queue.size();
    if (i) s += ",";
    s += (t.window > 0 ? "sliding:" : "full:") + std::to_string(used) + "/" +
         std::to_string(t.pool.num_blocks);
  }
  if (capacity > 0) {
    const int64_t n = (int64_t)s.size() < capacity - 1 ? (int64_t)s.size() : capacity - 1;
    std::memcpy(buf, s.data(), n);
    buf[n] = '\0';
  }
  return (int64_t)s.size();
}

int pkv_manager_block_table(const pkv_kv_manager* mgr, int32_t type, const int64_t* request_ids,
                            int32_t B, int32_t max_blocks_per_seq, int32_t* table_out) {
  PKV_REQUIRE(mgr && type >= 0 && type < (int32_t)mgr->types.size() && B >= 0 &&
                  max_blocks_per_seq > 0 && (B == 0 || (request_ids && table_out)),
              PKV_ERR_INVALID_ARG, "pkv_manager_block_table: bad args");
  const pkv::TypeManager& t = mgr->types[type];
  for (int32_t b = 0; b < B; ++b) {
    auto it = t.req_blocks.find(request_ids[b]);
    const int64_t n = it == t.req_blocks.end() ? 0 : (int64_t)it->second.size();
    PKV_REQUIRE(n <= max_blocks_per_seq, PKV_ERR_INVALID_ARG,
                "pkv_manager_block_table: request %lld holds %lld blocks > %d",
                (long long)request_ids[b], (long long)n, max_blocks_per_seq);
  }
  for (int32_t b = 0; b < B; ++b) {
    int32_t* row = table_out + (int64_t)b * max_blocks_per_seq;
    auto it = t.req_blocks.find(request_ids[b]);
    int64_t j = 0;
    if (it != t.req_blocks.end())
      for (; j < (int64_t)it->second.size(); ++j) row[j] = it->second[j];
    for (; j < max_blocks_per_seq; ++j) row[j] = t.null();
  }
  return PKV_OK;
}

uint64_t pkv_block_hash(uint64_t parent_hash, int32_t has_parent, const int32_t* tokens,
                        int32_t num_tokens, int32_t group_id) {
  if (num_tokens < 0 || (num_tokens > 0 && !tokens)) return 0;
  return pkv::block_hash(parent_hash, has_parent != 0, tokens, num_tokens, group_id);
}

int64_t pkv_manager_match_prefix(pkv_kv_manager* mgr, int64_t request_id, const int32_t* tokens,
                                 int64_t num_tokens) {
  PKV_REQUIRE(mgr && num_tokens >= 0 && (tokens || num_tokens == 0), PKV_ERR_INVALID_ARG,
              "pkv_manager_match_prefix: bad args");
  for (const pkv::TypeManager& t : mgr->types)
    PKV_REQUIRE(t.held(request_id) == 0, PKV_ERR_INVALID_ARG,
                "pkv_manager_match_prefix: request %lld already holds blocks",
                (long long)request_id);
  for (const pkv::TypeManager& t : mgr->types)
    if (t.window > 0 || !t.prefix) return 0;
  std::vector<std::vector<int32_t>> hits;
  size_t n = SIZE_MAX;
  for (const pkv::TypeManager& t : mgr->types) {
    hits.push_back(t.match(tokens, num_tokens));
    if (hits.back().size() < n) n = hits.back().size();
  }
  if (n == 0) return 0;
  for (size_t i = 0; i < mgr->types.size(); ++i) {
    pkv::TypeManager& t = mgr->types[i];
    std::vector<int32_t> blocks(hits[i].begin(), hits[i].begin() + n);
    for (int32_t b : blocks) ++t.pool.ref[b];
    t.req_blocks[request_id] = blocks;
    t.req_hashes[request_id] = t.chain(tokens, (int64_t)n);
  }
  return (int64_t)n * mgr->block_size;
}

int pkv_manager_cache_blocks(pkv_kv_manager* mgr, int64_t request_id, const int32_t* tokens,
                             int64_t num_tokens) {
  PKV_REQUIRE(mgr && num_tokens >= 0 && (tokens || num_tokens == 0), PKV_ERR_INVALID_ARG,
              "pkv_manager_cache_blocks: bad args");
  for (pkv::TypeManager& t : mgr->types) t.cache_full_blocks(request_id, tokens, num_tokens);
  return PKV_OK;
}

int64_t pkv_manager_fork(pkv_kv_manager* mgr, int64_t parent_id, const int64_t* child_ids,
                         int32_t num_children, int64_t num_tokens, int32_t shareable,
                         int32_t* copy_src, int32_t* copy_dst, int64_t capacity,
                         int64_t* copies_per_type) {
  PKV_REQUIRE(mgr && num_children >= 0 && (child_ids || num_children == 0) && num_tokens >= 0 &&
                  capacity >= 0 && ((copy_src && copy_dst) || capacity == 0) && copies_per_type,
              PKV_ERR_INVALID_ARG, "pkv_manager_fork: bad args");
  const int64_t bs = mgr->block_size;
  const int64_t nblk = pkv::ceil_div(num_tokens, bs), n_full = num_tokens / bs;
  // Plan and check everything before changing anything.
  int64_t total = 0;
  for (size_t i = 0; i < mgr->types.size(); ++i) {
    const pkv::TypeManager& t = mgr->types[i];
    PKV_REQUIRE(t.held(parent_id) >= nblk, PKV_ERR_INVALID_ARG,
                "pkv_manager_fork: parent %lld holds fewer than %lld blocks", (long long)parent_id,
                (long long)nblk);
    const std::vector<int32_t>& row = t.req_blocks.at(parent_id);
    int64_t copies = 0;
    for (int64_t j = 0; j < nblk; ++j)
      copies += row[j] != t.null() && !(shareable && j < n_full);
    copies *= num_children;
    PKV_REQUIRE((int64_t)t.pool.queue.size() >= copies, PKV_ERR_OUT_OF_BLOCKS,
                "pkv_manager_fork: type %zu needs %lld blocks, %lld free", i, (long long)copies,
                (long long)t.pool.queue.size());
    total += copies;
  }
  PKV_REQUIRE(total <= capacity, PKV_ERR_INVALID_ARG,
              "pkv_manager_fork: %lld copies do not fit capacity %lld", (long long)total,
              (long long)capacity);
  for (int32_t c = 0; c < num_children; ++c)
    for (const pkv::TypeManager& t : mgr->types)
      PKV_REQUIRE(child_ids[c] != parent_id && t.held(child_ids[c]) == 0, PKV_ERR_INVALID_ARG,
                  "pkv_manager_fork: child %lld already holds blocks", (long long)child_ids[c]);
  int64_t k = 0;
  for (size_t i = 0; i < mgr->types.size(); ++i) {
    pkv::TypeManager& t = mgr->types[i];
    const std::vector<int32_t> prow(t.req_blocks.at(parent_id).begin(),
                                    t.req_blocks.at(parent_id).begin() + nblk);
    const int64_t k0 = k;
    for (int32_t c = 0; c < num_children; ++c) {
      std::vector<int32_t> row;
      row.reserve(nblk);
      for (int64_t j = 0; j < nblk; ++j) {
        const int32_t b = prow[j];
        if (b == t.null()) {
          row.push_back(b);
        } else if (shareable && j < n_full) {
          ++t.pool.ref[b];
          row.push_back(b);
        } else {
          int32_t nb;
          pkv::pool_take(&t.pool, 1, &nb);
          copy_src[k] = b;
          copy_dst[k] = nb;
          ++k;
          row.push_back(nb);
        }
      }
      t.req_blocks[child_ids[c]] = std::move(row);
      if (shareable && t.prefix) {
        auto ph = t.req_hashes.find(parent_id);
        if (ph != t.req_hashes.end()) {
          const size_t nh = ph->second.size() < (size_t)n_full ? ph->second.size() : (size_t)n_full;
          t.req_hashes[child_ids[c]] = std::vector<uint64_t>(ph->second.begin(), ph->second.begin() + nh);
        }
      }
    }
    copies_per_type[i] = k - k0;
  }
  return k;
}

}  // extern "C"
