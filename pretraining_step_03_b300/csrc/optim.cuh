// Per-matrix table entry of the Muon kernels (device-resident array).
#pragma once

namespace nc {

struct MuonMat {
    long off;     // element offset of the matrix in the flat parameter / grad / momentum arrays
    long x_off;   // element offset of its (wide-oriented) X in the Newton-Schulz buffer
    int rows, cols;
    int tr;       // 1: rows > cols, X holds the transpose
    float scale;  // sqrt(max(1, rows/cols))
};

}  // namespace nc
