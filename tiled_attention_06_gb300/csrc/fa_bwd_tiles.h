// Tile geometry shared by the backward kernels (fa_backward.cu) and the host code that
// encodes their tensor maps (fa_api.cu).
#pragma once

namespace fa {

// Rows of one TMA box of the backward's tensor maps (Q, dO, K, V): the streamed side of each
// backward kernel moves in 64-row halves, and a resident 128-row tile is loaded as two boxes.
constexpr int kBwdBoxRows = 64;

}  // namespace fa
