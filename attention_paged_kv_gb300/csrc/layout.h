// Plan metadata layout shared by the host planner and the kernels (int32
// words; every region 256-byte aligned).  Host-safe: no device code.
#pragma once

#include <cstdint>

namespace pa {

enum HdrIdx : int {
  H_MAGIC = 0, H_VERSION, H_B, H_HQ, H_HKV, H_D, H_PS, H_NUM_PAGES, H_DTYPE, H_CAUSAL,
  H_T, H_NNZ, H_NDEC, H_NPRE, H_NMERGE, H_NPART, H_DEC_CHUNK, H_PRE_CHUNK, H_NUM_SMS, H_G,
  H_OFF_PAGES, H_OFF_REQ, H_OFF_DEC, H_OFF_PRE, H_OFF_MERGE, H_BLOB_BYTES, H_OFF_PART_O,
  H_OFF_PART_LSE, H_TOTAL_BYTES, H_DEC_CORES,
  H_STATUS = 32,
  H_NDEC_CLASS0 = 33,  // decode items per row class (<= 8, 16, 32, 64 rows), in item order
  H_LAYOUT = 37,       // cache layout: 0 NHD, 1 HND
  H_NGROUPS = 38,      // shared-prefix groups (request entries B .. B + groups - 1 are their prefixes)
  H_PRE_TILES = 39,    // 128-row Q tiles per prefill item (1 or 2)
  HDR_WORDS = 64
};

constexpr int32_t kMagic = 0x50414731;
constexpr int32_t kVersion = 5;
constexpr int kDecClasses = 4;
constexpr int kDecMaxRows = 32;  // packed (token, head) rows of a small-query item
constexpr int kQRows = 128;   // packed query rows per prefill MMA tile
constexpr int kItemRows = 256;  // packed query rows per prefill work item (two tiles)
constexpr int kKvTile = 128;  // keys per prefill key tile

struct ReqEntry { int32_t qo_start, qo_len, kv_len, page_start; };
struct DecItem { int32_t req, kv_head, tok0, tok1, part_row, page_start, pad1, pad2; };  // page_start: req's
struct PreItem { int32_t req, kv_head, q_tok0, q_ntok, kv_tok0, kv_tok1, part_row, pad0; };
struct MergeEntry { int32_t out_row0, part_row0, nsplit, split_stride; };
static_assert(sizeof(DecItem) == 32 && sizeof(PreItem) == 32 && sizeof(MergeEntry) == 16, "layout");

}  // namespace pa
