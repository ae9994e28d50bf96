// Host-side block management: BlockPool, block tables and slot_mapping.
//
// Follows "KV Cache 管理设计文档": §2.4 BlockPool (FIFO queue + set, first popped
// id is the null block), §2.3 / §2.3.2 skipped tokens and null-padded sliding
// tables, §4.2.1 calculate_block_num, §4.2.2 prepare_block_tables /
// prepare_slot_mapping; and "KVCache 优化技能" §3.1-3.3 for the slot formula and
// the static arange table.
#include <cstring>
#include <vector>

#include "abi_common.h"
#include "host_pool.h"

namespace pkv {

static thread_local std::string g_last_error;

void set_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
}

void clear_error() { g_last_error.clear(); }

}  // namespace pkv

extern "C" {

const char* pkv_last_error(void) { return pkv::g_last_error.c_str(); }

int pkv_version(void) { return 100; }

int pkv_pool_create(int64_t num_blocks, const int32_t* initial_order, pkv_pool** out) {
  PKV_REQUIRE(out != nullptr, PKV_ERR_INVALID_ARG, "pkv_pool_create: out is NULL");
  PKV_REQUIRE(num_blocks >= 1 && num_blocks <= INT32_MAX, PKV_ERR_INVALID_ARG,
              "pkv_pool_create: num_blocks %lld out of range", (long long)num_blocks);
  auto* p = new pkv_pool();
  p->num_blocks = num_blocks;
  std::vector<uint8_t> seen(num_blocks, 0);
  for (int64_t i = 0; i < num_blocks; ++i) {
    int32_t id = initial_order ? initial_order[i] : (int32_t)i;
    if (id < 0 || id >= num_blocks || seen[id]) {
      delete p;
      PKV_FAIL(PKV_ERR_INVALID_ARG, "pkv_pool_create: initial_order is not a permutation");
    }
    seen[id] = 1;
    p->queue.push_back(id);
  }
  p->ref.assign(num_blocks, 0);
  p->null_block = p->queue.front();  // first popped id: the placeholder block
  p->queue.pop_front();
  *out = p;
  pkv::clear_error();
  return PKV_OK;
}

void pkv_pool_destroy(pkv_pool* pool) { delete pool; }

int32_t pkv_pool_null_block(const pkv_pool* pool) { return pool ? pool->null_block : -1; }

int64_t pkv_pool_num_free(const pkv_pool* pool) { return pool ? (int64_t)pool->queue.size() : -1; }

int pkv_pool_alloc(pkv_pool* pool, int64_t n, int32_t* ids_out) {
  PKV_REQUIRE(pool && (n == 0 || ids_out) && n >= 0, PKV_ERR_INVALID_ARG, "pkv_pool_alloc: bad args");
  PKV_REQUIRE((int64_t)pool->queue.size() >= n, PKV_ERR_OUT_OF_BLOCKS,
              "pkv_pool_alloc: need %lld blocks, %lld free", (long long)n,
              (long long)pool->queue.size());
  pkv::pool_take(pool, n, ids_out);
  return PKV_OK;
}

int pkv_pool_free(pkv_pool* pool, const int32_t* ids, int64_t n) {
  PKV_REQUIRE(pool && (n == 0 || ids) && n >= 0, PKV_ERR_INVALID_ARG, "pkv_pool_free: bad args");
  // Validate everything first so that a failing call leaves the pool unchanged.
  PKV_REQUIRE(pkv::pool_release_ok(pool, ids, n), PKV_ERR_DOUBLE_FREE,
              "pkv_pool_free: an id is out of range, the null block, or released more often "
              "than it is referenced");
  pkv::pool_release(pool, ids, n, nullptr);
  return PKV_OK;
}

int pkv_pool_share(pkv_pool* pool, const int32_t* ids, int64_t n) {
  PKV_REQUIRE(pool && (n == 0 || ids) && n >= 0, PKV_ERR_INVALID_ARG, "pkv_pool_share: bad args");
  for (int64_t i = 0; i < n; ++i) {
    const int32_t id = ids[i];
    PKV_REQUIRE(id >= 0 && id < pool->num_blocks && id != pool->null_block && pool->ref[id] > 0,
                PKV_ERR_INVALID_ARG, "pkv_pool_share: block %d is not held", id);
  }
  for (int64_t i = 0; i < n; ++i) ++pool->ref[ids[i]];
  return PKV_OK;
}

int32_t pkv_pool_ref_count(const pkv_pool* pool, int32_t id) {
  if (!pool || id < 0 || id >= pool->num_blocks) return -1;
  return pool->ref[id];
}

int64_t pkv_num_skipped_tokens(int64_t num_computed_tokens, int64_t window) {
  if (window <= 0) return 0;
  int64_t s = num_computed_tokens - window + 1;
  return s > 0 ? s : 0;
}

int pkv_build_block_table(pkv_pool* pool, const int32_t* seq_lens, int32_t B, int32_t block_size,
                          int32_t window, int32_t max_blocks_per_seq, int32_t* table_out) {
  PKV_REQUIRE(pool && seq_lens && table_out && B >= 0 && block_size > 0 && max_blocks_per_seq > 0,
              PKV_ERR_INVALID_ARG, "pkv_build_block_table: bad args");
  // Plan every row first (all-or-nothing on the pool).
  std::vector<int64_t> n_null(B), n_live(B);
  int64_t need = 0;
  for (int32_t b = 0; b < B; ++b) {
    PKV_REQUIRE(seq_lens[b] >= 0, PKV_ERR_INVALID_ARG, "pkv_build_block_table: negative length");
    int64_t nblk = pkv::ceil_div(seq_lens[b], block_size);
    PKV_REQUIRE(nblk <= max_blocks_per_seq, PKV_ERR_INVALID_ARG,
                "pkv_build_block_table: sequence %d needs %lld blocks > max_blocks_per_seq %d", b,
                (long long)nblk, max_blocks_per_seq);
    int64_t skipped = seq_lens[b] > 0 ? pkv_num_skipped_tokens(seq_lens[b] - 1, window) : 0;
    int64_t nn = skipped / block_size;
    if (nn > nblk) nn = nblk;
    n_null[b] = nn;
    n_live[b] = nblk - nn;
    need += n_live[b];
  }
  PKV_REQUIRE((int64_t)pool->queue.size() >= need, PKV_ERR_OUT_OF_BLOCKS,
              "pkv_build_block_table: need %lld blocks, %lld free", (long long)need,
              (long long)pool->queue.size());
  for (int32_t b = 0; b < B; ++b) {
    int32_t* row = table_out + (int64_t)b * max_blocks_per_seq;
    int64_t j = 0;
    for (; j < n_null[b]; ++j) row[j] = pool->null_block;
    pkv::pool_take(pool, n_live[b], row + j);
    j += n_live[b];
    for (; j < max_blocks_per_seq; ++j) row[j] = pool->null_block;
  }
  return PKV_OK;
}

int pkv_build_block_table_arange(int32_t B, int32_t blocks_per_seq, int32_t* table_out) {
  PKV_REQUIRE(table_out && B >= 0 && blocks_per_seq > 0, PKV_ERR_INVALID_ARG,
              "pkv_build_block_table_arange: bad args");
  for (int64_t i = 0; i < (int64_t)B * blocks_per_seq; ++i) table_out[i] = (int32_t)i;
  return PKV_OK;
}

int64_t pkv_build_slot_mapping(const int32_t* block_table, int32_t max_blocks_per_seq,
                               const int32_t* start_pos, const int32_t* num_new, int32_t B,
                               int32_t block_size, int32_t* slots_out, int64_t slots_capacity) {
  PKV_REQUIRE(block_table && start_pos && num_new && B >= 0 && block_size > 0 &&
                  max_blocks_per_seq > 0 && (slots_out || slots_capacity == 0),
              PKV_ERR_INVALID_ARG, "pkv_build_slot_mapping: bad args");
  int64_t t = 0;
  for (int32_t b = 0; b < B; ++b) {
    PKV_REQUIRE(start_pos[b] >= 0 && num_new[b] >= 0, PKV_ERR_INVALID_ARG,
                "pkv_build_slot_mapping: negative position or count (sequence %d)", b);
    for (int32_t i = 0; i < num_new[b]; ++i, ++t) {
      int64_t pos = (int64_t)start_pos[b] + i;
      int64_t lb = pos / block_size;
      PKV_REQUIRE(lb < max_blocks_per_seq, PKV_ERR_INVALID_ARG,
                  "pkv_build_slot_mapping: position %lld beyond the table (sequence %d)",
                  (long long)pos, b);
      PKV_REQUIRE(t < slots_capacity, PKV_ERR_INVALID_ARG,
                  "pkv_build_slot_mapping: slots_out too small");
      int64_t pb = block_table[(int64_t)b * max_blocks_per_seq + lb];
      int64_t slot = pb * block_size + pos % block_size;
      PKV_REQUIRE(pb >= 0 && slot <= INT32_MAX, PKV_ERR_INVALID_ARG,
                  "pkv_build_slot_mapping: slot does not fit int32");
      slots_out[t] = (int32_t)slot;
    }
  }
  return t;
}

int64_t pkv_block_num_fixed(int64_t max_concurrency, int64_t sliding_window, int64_t next_n,
                            int64_t block_size) {
  return max_concurrency * (pkv::ceil_div(sliding_window + 2 * next_n, block_size) + 1) + 1;
}

int64_t pkv_block_num_full_offline(int64_t max_len, int64_t block_size, int64_t max_concurrency) {
  return pkv::ceil_div(max_len, block_size) * max_concurrency + 1;
}

int64_t pkv_block_num_full_online(int64_t available_bytes, int64_t per_token_bytes,
                                  int64_t block_size) {
  if (per_token_bytes <= 0 || block_size <= 0) return -1;
  return (available_bytes / per_token_bytes) / block_size + 1;
}

}  // extern "C"
