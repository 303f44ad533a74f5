// cascade_plan.h -- layout of the shared-prefix work plan that
// pkv_plan_shared_prefix writes (host) and pa_cascade_kernel reads (device).
//
// The plan is one int32 array:
//   header[kHeader]            see the H_* indices
//   expected[num_seqs]         partials each sequence receives (one per item
//                              that holds its rows)
//   counters[num_seqs * Hk]    arrivals per (sequence, kv head); zero between
//                              calls (the kernel that merges resets them)
//   items[num_items][item_ints]
// An item is {seq0, nrows, slot, nseg, then nseg segments of {table_seq,
// tok_begin, tok_end, row_lo, row_hi}}: query rows r < nrows are head
// r % G of sequence seq0 + r / G; segment k covers tokens [tok_begin,
// tok_end) addressed by table_seq's block table, for rows [row_lo, row_hi).
// nseg == 0 marks a sequence with an empty or invalid context (zero output).
#pragma once

namespace pkv {
namespace plan {

constexpr int kHeader = 8;
enum : int {
    H_NUM_ITEMS = 0,
    H_SLOTS = 1,
    H_NUM_SEQS = 2,
    H_NUM_KV_HEADS = 3,
    H_ITEM_INTS = 4,
    H_MAX_SEG = 5,
    H_PARTITION = 6,
    H_TAG = 7,
};
constexpr int kTag = 0x43564b50;    // "PKVC"
constexpr int kNT = 3;              // n-tiles of 8 query rows per item
constexpr int kMaxRows = 8 * kNT;   // query rows per item
constexpr int kItemHead = 4;
// Block-table entries one item may address (all segments together): the
// planner keeps items within it and the kernel stages that many.
constexpr int kTableCap = 256;
constexpr int kSegInts = 5;

constexpr int max_segments(int group) { return 1 + kMaxRows / group; }
constexpr int item_ints(int group) { return kItemHead + kSegInts * max_segments(group); }

}  // namespace plan
}  // namespace pkv
