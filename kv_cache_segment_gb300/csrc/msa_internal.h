// msa_internal.h -- data shared by the host planner and the CUDA kernels of
// libmsa (work items, output groups, segment runs, workspace layout).
// Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

namespace msa {

constexpr int kBlock = 16;       // tokens per KV block (the only supported size)
constexpr int kTileKeys = 128;   // keys per KV tile staged in shared memory
constexpr int kTileRows = 128;   // query rows per prefill tile (tcgen05 M)
constexpr int kDecRows = 16;     // MMA rows of a decode item (query rows x G heads)

enum ItemKind : int32_t { kDecode = 0, kPrefill = 1 };

// A physically contiguous segment of one sequence, in tokens:
// logical keys [log_start, log_start + n_tok) live in pool rows
// [phys_row, phys_row + n_tok).
struct Run {
    int32_t log_start;
    int32_t phys_row;
    int32_t n_tok;
    int32_t pad;
};

// An output group: the rows and heads one merge produces.
//   decode : rows [row0, row0+nrows) x query heads [head*G, head*G+G), kv head = head
//   prefill: `pad` query tiles of 128 rows x one head, all of one kv head:
//            pad == 2, nrows <= 128: rows [row0, row0+nrows) x heads
//                    [head, head+2) (every head for even G, all but the
//                    last of each kv head for odd G);
//            otherwise (the last query head of a kv head, odd G): head
//                    `head` x rows [row0, row0+nrows) (<= 128 * pad),
//                    tile k = rows [row0 + 128k, ...)
// n_parts > 1 means the key range was split; parts write partials to slots
// [slot, slot + n_parts) (two tile slots each for prefill) and the last to
// finish merges them.
struct Group {
    int32_t kind;
    int32_t seq;
    int32_t head;
    int32_t row0;
    int32_t nrows;
    int32_t n_parts;
    int32_t slot;
    int32_t pad;  // decode: G query heads; prefill: query tiles (1 or 2)
};

// A work item: one group's keys [kb, ke), starting in run `first_run`
// (global run index).
struct Item {
    int32_t group;
    int32_t kb;
    int32_t ke;
    int32_t first_run;
    int32_t part;
    int32_t kind;
    int32_t seq;
    int32_t pad;  // number of KV tiles the item walks (filled by the planner)
};

// Byte offsets of the sections of the device workspace.
struct WsLayout {
    size_t error;       // int32[64]: [0] error word, rest reserved
    size_t items;       // Item[n_items]
    size_t groups;      // Group[n_groups]
    size_t runs;        // Run[n_runs]
    size_t pos;         // int32[n_q]: logical position of each packed row
    size_t order;       // int32[n_items]: item ids in processing order (longest first)
    size_t image_end;   // end of the part copied from the host image
    size_t counters;    // int32[2 * n_groups]: merge arrival counters per head slot (zeroed)
    size_t sched;       // int32[2]: queue head, CTAs finished (zeroed; the last CTA resets them)
    size_t counters_end;
    size_t dec_part;    // float[n_dec_slots][kDecRows][D]
    size_t dec_lse;     // float[n_dec_slots][kDecRows]
    size_t pre_part;    // float[n_pre_slots][2][kTileRows][D]
    size_t pre_lse;     // float[n_pre_slots][2][kTileRows]
    size_t total;
};

// Error word codes written by kernels (bit flags, OR-ed); the public names
// are the MSA_DEVERR_* constants of msa.h.
enum DeviceError : int32_t {
    kErrTimeoutProducer = 1 << 0,
    kErrTimeoutMma = 1 << 1,
    kErrTimeoutCompute = 1 << 2,
    kErrBadIndex = 1 << 3,
    kErrAppendSlot = 1 << 4,
    kErrTmemAlloc = 1 << 5,
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace msa
