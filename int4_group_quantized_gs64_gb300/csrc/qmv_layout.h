// qmv_layout.h - sizes that the decode kernels and the workspace layouts
// share (kept apart from the launcher declarations so that a kernel's
// dependencies are exactly its source and the headers it compiles).
#pragma once

namespace qmv {

// Stage-level work split of the tensor-map decode kernels: CTAs of one
// launch at most, and per CTA the partial-sum slots of the items it shares
// with other CTAs (2 slots x 256 rows x 8 tokens).
constexpr int kSkMaxCtas = 256;
constexpr int kSkPartFloats = 2 * 256 * 8;

// Pass-packed activation units (tensor-map decode path, in that kernel's
// int4 form): block (pi, s) of kPackedStage bytes holds, for pass pi and
// stage s (4 groups), the records (power-of-two factor, offset_init) of the
// pass's token slots 0..7 ([slot][4] float2, 256 B) followed by their units
// ([slot][4 groups x 16] uint4, 1 KB a slot), so a stage's activations are
// one contiguous copy of 256 B + 1 KB per token.
constexpr int kPackedHead = 8 * 4 * 8;
constexpr int kPackedStage = kPackedHead + 8 * 1024;

}  // namespace qmv
