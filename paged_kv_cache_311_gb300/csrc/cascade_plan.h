// cascade_plan.h -- layout of the shared-prefix work plan that
// pkv_plan_shared_prefix writes (host) and pa_cascade_kernel and
// pa_cascade_merge_kernel read (device).
//
// The plan is one int32 array, read-only for the device:
//   header[kHeader]            see the H_* indices
//   expected[num_seqs]         partials each sequence receives (one per item
//                              that holds its rows; 1: the item writes the
//                              output itself; 0: empty or invalid context)
//   lens[num_seqs]             the context lengths the plan was made for (the
//                              kernel rejects a sequence whose device length
//                              differs)
//   items[num_items][item_ints]
// One CTA per (kv head, list) works through the items of its list: list k
// starts at item k and follows the items' next links (-1 ends it; a link
// always points further down the array).  An item is {seq0, nrows, slot,
// nseg, tiles, ids, checks, next}, then kMaxRows member sequence ids, then
// max_segments segments of {table_seq, tok_begin, tok_end, row_lo, row_hi,
// first_tile, id_off, check_off}, then kTableCap block ids: query rows
// r < nrows are head r % G of sequence members[r / G] (a group's members
// need not be neighbours in the batch; seq0 is the first member); segment k
// covers tokens [tok_begin, tok_end) addressed by table_seq's block table,
// for rows [row_lo, row_hi); its 16-token tiles are the item's tiles
// [first_tile, ...), its block ids start at id_off, and its device-table
// checks (one per block, per member for a shared-prefix segment) at
// check_off; tiles, ids and checks are the item's totals.  The block ids are
// the physical blocks of the segments' logical blocks [tok_begin / bs,
// ceil(tok_end / bs)), segment after segment, as the host tables held them
// when the plan was made (the kernel starts its loads from them and checks
// the device tables meanwhile).  nseg == 0 marks a sequence with an empty or
// invalid context (zero output).
#pragma once

namespace pkv {
namespace plan {

constexpr int kHeader = 8;
enum : int {
    H_NUM_LISTS = 0,     // work lists: one CTA per (kv head, list)
    H_SLOTS = 1,
    H_NUM_SEQS = 2,
    H_NUM_KV_HEADS = 3,
    H_ITEM_INTS = 4,
    H_MAX_SEG = 5,
    H_TARGET = 6,        // target tokens per list the plan was cut with
    H_NUM_ITEMS = 7,
};
constexpr int kNT = 3;              // n-tiles of 8 query rows per item
constexpr int kMaxRows = 8 * kNT;   // query rows per item
constexpr int kItemHead = 8;
enum : int { I_SEQ0 = 0, I_NROWS, I_SLOT, I_NSEG, I_TILES, I_IDS, I_CHECKS, I_NEXT };
enum : int { S_TABLE_SEQ = 0, S_BEGIN, S_END, S_ROW_LO, S_ROW_HI, S_FIRST_TILE, S_ID_OFF, S_CHECK_OFF };
// Block-table entries one item may address (all segments together): the
// planner keeps items within it and the kernel stages that many.
constexpr int kTableCap = 256;
constexpr int kSegInts = 8;
constexpr int kTileTokens = 16;     // tokens per warp tile of the kernel

constexpr int max_segments(int group) { return 1 + kMaxRows / group; }
constexpr int item_segments_offset() { return kItemHead + kMaxRows; }
constexpr int item_ids_offset(int group) { return item_segments_offset() + kSegInts * max_segments(group); }
constexpr int item_ints(int group) { return item_ids_offset(group) + kTableCap; }

}  // namespace plan

// How the shared-prefix kernel that the current engine choice runs takes a
// plan (the planner's automatic cut follows it): resident CTAs per SM (3 for
// the warp-level kernel, 1 for the tcgen05 kernel) and what a CTA's switch
// from one item to the next costs in 16-token tiles streamed.  The engine
// choice (pkv_decode_set_engine) passes its value on with
// set_shared_plan_engine.  Defined in pkv_plan.cu.
void set_shared_plan_engine(int engine);
int shared_ctas_per_sm(int head_dim);
int shared_item_cost_tiles(int head_dim);

}  // namespace pkv
