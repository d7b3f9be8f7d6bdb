// qr_capi.cu -- the extern "C" entry points of libqr.so (declared in
// include/qr.h): host-side argument validation, then a launch on the
// caller's stream.  Validation runs before any CUDA call, so a rejected call
// touches neither memory nor the device.
//
// Checks, in this order (the first failure is returned):
//   1. null pointers, n == 0, R < 1                        -> QR_ERR_INVALID_ARG
//   2. bits not in {3,4,6,8}, unknown dtype, R > 8         -> QR_ERR_UNSUPPORTED
//   3. a byte count overflowing size_t                     -> QR_ERR_SIZE
//   4. a device pointer not 16-byte aligned                -> QR_ERR_MISALIGNED
//   5. an output partially overlapping another buffer      -> QR_ERR_INVALID_ARG
// A launch error reported by the runtime                   -> QR_ERR_CUDA
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/qr.h"
#include "qr_launch.h"

#define QR_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kTile = 2048;

bool bits_ok(int bits) { return bits == 3 || bits == 4 || bits == 6 || bits == 8; }
bool dtype_ok(qr_dtype_t d) { return d == QR_FP16 || d == QR_BF16; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t tile_bytes(int bits) { return bits_ok(bits) ? size_t(256) * size_t(bits) + 128 : 0; }

// ceil(n/2048) * tile_bytes, or 0 on overflow
size_t wire_bytes(int bits, size_t n) {
    const size_t tb = tile_bytes(bits);
    if (tb == 0) return 0;
    const size_t tiles = n / kTile + (n % kTile != 0);
    if (tiles > SIZE_MAX / tb) return 0;
    return tiles * tb;
}

// the 16-bit value buffers of n values: 2n bytes, and n must index as long long
bool value_bytes_ok(size_t n) { return n <= (SIZE_MAX / 4); }

// [a, a+na) and [b, b+nb) share a byte
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// an output may equal an input exactly (in place) but not overlap it partially
bool bad_alias(const void *out, size_t nout, const void *in, size_t nin) {
    return out != in && overlaps(out, nout, in, nin);
}

qr_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? QR_OK : QR_ERR_CUDA; }

}  // namespace


QR_EXPORT size_t qr_tile_values(void) { return kTile; }

QR_EXPORT size_t qr_tile_bytes(int bits) { return tile_bytes(bits); }

QR_EXPORT size_t qr_wire_bytes(int bits, size_t n) { return wire_bytes(bits, n); }

namespace {

// R*(R+1)*ceil(ceil(n/2048)/R) tiles, 0 on overflow or bad arguments
size_t twoshot_ws_bytes(int bits, int R, size_t n) {
    const size_t tb = tile_bytes(bits);
    if (tb == 0 || R < 1 || R > QR_MAX_RANKS) return 0;
    const size_t tiles = n / kTile + (n % kTile != 0);
    const size_t seg = tiles / size_t(R) + (tiles % size_t(R) != 0);
    const size_t bufs = size_t(R) * size_t(R + 1);
    if (seg > SIZE_MAX / bufs || seg * bufs > SIZE_MAX / tb) return 0;
    return seg * bufs * tb;
}

}  // namespace

QR_EXPORT size_t qr_twoshot_workspace_bytes(int bits, int R, size_t n) { return twoshot_ws_bytes(bits, R, n); }

namespace {

// The two-shot workspace, then (16-byte aligned) 2T + 1 flag words.
size_t twoshot_flags_ws_bytes(int bits, int R, size_t n, size_t *flags_offset) {
    const size_t base = twoshot_ws_bytes(bits, R, n);
    if (base == 0) return 0;
    const size_t tiles = n / kTile + (n % kTile != 0);
    const size_t off = (base + 15) / 16 * 16;
    if (tiles > (SIZE_MAX - off) / 8 - 1) return 0;
    if (flags_offset) *flags_offset = off;
    return off + (2 * tiles + 1) * sizeof(uint32_t);
}

}  // namespace

QR_EXPORT size_t qr_twoshot_flags_workspace_bytes(int bits, int R, size_t n) {
    return twoshot_flags_ws_bytes(bits, R, n, nullptr);
}

// qr_allreduce_twoshot_flags and its self-test share the checks and the launch.
static qr_status_t twoshot_flags_call(int bits, qr_dtype_t dtype, int R, const void *const *x, size_t n,
                                      void *const *y, void *workspace, size_t workspace_bytes, int drop_sender,
                                      qr_stream_t stream) {
    if (!x || !y || !workspace || n == 0 || R < 1) return QR_ERR_INVALID_ARG;
    for (int r = 0; r < R && r < QR_MAX_RANKS; ++r)
        if (!x[r] || !y[r]) return QR_ERR_INVALID_ARG;
    if (!bits_ok(bits) || !dtype_ok(dtype) || R > QR_MAX_RANKS) return QR_ERR_UNSUPPORTED;
    size_t flags_offset = 0;
    const size_t need = twoshot_flags_ws_bytes(bits, R, n, &flags_offset);
    if (!value_bytes_ok(n) || need == 0 || wire_bytes(bits, n) == 0) return QR_ERR_SIZE;
    if (workspace_bytes < need) return QR_ERR_SIZE;
    const size_t V = 2 * n;
    if (!aligned16(workspace)) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r)
        if (!aligned16(x[r]) || !aligned16(y[r])) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r) {
        if (overlaps(workspace, need, x[r], V) || overlaps(workspace, need, y[r], V)) return QR_ERR_INVALID_ARG;
        for (int i = 0; i < R; ++i) {
            // tile t of every input is read before tile t of any output is
            // written: an output may be an input exactly, never partly
            if (bad_alias(y[r], V, x[i], V)) return QR_ERR_INVALID_ARG;
            if (i < r && overlaps(y[r], V, y[i], V)) return QR_ERR_INVALID_ARG;
        }
    }
    return from_cuda(qrk::launch_twoshot_flags(bits, dtype, R, x, static_cast<long long>(n), y, workspace,
                                               static_cast<uint8_t *>(workspace) + flags_offset, drop_sender,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

QR_EXPORT qr_status_t qr_allreduce_twoshot_flags(int bits, qr_dtype_t dtype, int R, const void *const *x, size_t n,
                                                 void *const *y, void *workspace, size_t workspace_bytes,
                                                 qr_stream_t stream) {
    return twoshot_flags_call(bits, dtype, R, x, n, y, workspace, workspace_bytes, -1, stream);
}

QR_EXPORT qr_status_t qr_selftest_twoshot_flags_drop(int bits, qr_dtype_t dtype, int R, const void *const *x,
                                                     size_t n, void *const *y, void *workspace,
                                                     size_t workspace_bytes, int drop_sender, qr_stream_t stream) {
    if (drop_sender < 0 || drop_sender >= R) return QR_ERR_INVALID_ARG;
    return twoshot_flags_call(bits, dtype, R, x, n, y, workspace, workspace_bytes, drop_sender, stream);
}

QR_EXPORT qr_status_t qr_allreduce_twoshot(int bits, qr_dtype_t dtype, int R, const void *const *x, size_t n,
                                           void *const *y, void *workspace, size_t workspace_bytes,
                                           qr_stream_t stream) {
    if (!x || !y || !workspace || n == 0 || R < 1) return QR_ERR_INVALID_ARG;
    for (int r = 0; r < R && r < QR_MAX_RANKS; ++r)
        if (!x[r] || !y[r]) return QR_ERR_INVALID_ARG;
    if (!bits_ok(bits) || !dtype_ok(dtype) || R > QR_MAX_RANKS) return QR_ERR_UNSUPPORTED;
    const size_t need = twoshot_ws_bytes(bits, R, n);
    if (!value_bytes_ok(n) || need == 0 || wire_bytes(bits, n) == 0) return QR_ERR_SIZE;
    if (workspace_bytes < need) return QR_ERR_SIZE;
    const size_t V = 2 * n;
    if (!aligned16(workspace)) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r)
        if (!aligned16(x[r]) || !aligned16(y[r])) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r) {
        if (overlaps(workspace, need, x[r], V) || overlaps(workspace, need, y[r], V)) return QR_ERR_INVALID_ARG;
        for (int i = 0; i < R; ++i) {
            // every input is read in Phase-1, before any output is written: an
            // output may be an input exactly (in place), never partly
            if (bad_alias(y[r], V, x[i], V)) return QR_ERR_INVALID_ARG;
            if (i < r && overlaps(y[r], V, y[i], V)) return QR_ERR_INVALID_ARG;
        }
    }
    return from_cuda(qrk::launch_twoshot(bits, dtype, R, x, static_cast<long long>(n), y, workspace,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

namespace {

bool fc_bits_ok(int bits) { return bits == 4 || bits == 8; }
bool fc_pair_ok(int rs, int ag) { return (rs == 4 && ag == 4) || (rs == 4 && ag == 8) || (rs == 8 && ag == 8); }

size_t fc_wire_bytes(int bits, size_t n) {
    if (!fc_bits_ok(bits)) return 0;
    const size_t tb = size_t(256) * size_t(bits) + 128;
    const size_t tiles = n / kTile + (n % kTile != 0);
    if (tiles > SIZE_MAX / tb) return 0;
    return tiles * tb;
}

}  // namespace

namespace {

// R*R*seg reduce-scatter tiles, then T all-gather tiles (0 on overflow or an
// unsupported pair or rank count).
size_t fc_twoshot_ws_bytes(int bits_rs, int bits_ag, int R, size_t n) {
    if (!fc_pair_ok(bits_rs, bits_ag) || R < 1 || R > QR_MAX_RANKS) return 0;
    const size_t tbi = size_t(256) * size_t(bits_rs) + 128, tbo = size_t(256) * size_t(bits_ag) + 128;
    const size_t tiles = n / kTile + (n % kTile != 0);
    const size_t seg = tiles / size_t(R) + (tiles % size_t(R) != 0);
    const size_t bufs = size_t(R) * size_t(R);
    if (seg > SIZE_MAX / bufs || seg * bufs > SIZE_MAX / tbi || tiles > SIZE_MAX / tbo) return 0;
    const size_t a = seg * bufs * tbi, b = tiles * tbo;
    if (a > SIZE_MAX - b) return 0;
    return a + b;
}

}  // namespace

QR_EXPORT size_t qr_fp4_twoshot_workspace_bytes(int R, size_t n) { return twoshot_ws_bytes(4, R, n); }

QR_EXPORT qr_status_t qr_fp4_allreduce_twoshot(qr_dtype_t dtype, int R, const void *const *x, size_t n,
                                               void *const *y, void *workspace, size_t workspace_bytes,
                                               qr_stream_t stream) {
    if (!x || !y || !workspace || n == 0 || R < 1) return QR_ERR_INVALID_ARG;
    for (int r = 0; r < R && r < QR_MAX_RANKS; ++r)
        if (!x[r] || !y[r]) return QR_ERR_INVALID_ARG;
    if (!dtype_ok(dtype) || R > QR_MAX_RANKS) return QR_ERR_UNSUPPORTED;
    const size_t need = twoshot_ws_bytes(4, R, n);
    if (!value_bytes_ok(n) || need == 0 || wire_bytes(4, n) == 0) return QR_ERR_SIZE;
    if (workspace_bytes < need) return QR_ERR_SIZE;
    const size_t V = 2 * n;
    if (!aligned16(workspace)) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r)
        if (!aligned16(x[r]) || !aligned16(y[r])) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r) {
        if (overlaps(workspace, need, x[r], V) || overlaps(workspace, need, y[r], V)) return QR_ERR_INVALID_ARG;
        for (int i = 0; i < R; ++i) {
            // every input is read in Phase-1, before any output is written: an
            // output may be an input exactly (in place), never partly
            if (bad_alias(y[r], V, x[i], V)) return QR_ERR_INVALID_ARG;
            if (i < r && overlaps(y[r], V, y[i], V)) return QR_ERR_INVALID_ARG;
        }
    }
    return from_cuda(qrk::launch_fp4_twoshot(dtype, R, x, static_cast<long long>(n), y, workspace,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

QR_EXPORT size_t qr_fc_twoshot_workspace_bytes(int bits_rs, int bits_ag, int R, size_t n) {
    return fc_twoshot_ws_bytes(bits_rs, bits_ag, R, n);
}

QR_EXPORT qr_status_t qr_fc_allreduce_twoshot(int bits_rs, int bits_ag, qr_dtype_t dtype, int R,
                                              const void *const *x, size_t n, void *const *y, void *workspace,
                                              size_t workspace_bytes, qr_stream_t stream) {
    if (!x || !y || !workspace || n == 0 || R < 1) return QR_ERR_INVALID_ARG;
    for (int r = 0; r < R && r < QR_MAX_RANKS; ++r)
        if (!x[r] || !y[r]) return QR_ERR_INVALID_ARG;
    if (!fc_pair_ok(bits_rs, bits_ag) || !dtype_ok(dtype) || R > QR_MAX_RANKS) return QR_ERR_UNSUPPORTED;
    const size_t need = fc_twoshot_ws_bytes(bits_rs, bits_ag, R, n);
    if (!value_bytes_ok(n) || need == 0) return QR_ERR_SIZE;
    if (workspace_bytes < need) return QR_ERR_SIZE;
    const size_t V = 2 * n;
    if (!aligned16(workspace)) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r)
        if (!aligned16(x[r]) || !aligned16(y[r])) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r) {
        if (overlaps(workspace, need, x[r], V) || overlaps(workspace, need, y[r], V)) return QR_ERR_INVALID_ARG;
        for (int i = 0; i < R; ++i) {
            // every input is read in Phase-1, before any output is written: an
            // output may be an input exactly (in place), never partly
            if (bad_alias(y[r], V, x[i], V)) return QR_ERR_INVALID_ARG;
            if (i < r && overlaps(y[r], V, y[i], V)) return QR_ERR_INVALID_ARG;
        }
    }
    return from_cuda(qrk::launch_fc_twoshot(bits_rs, bits_ag, dtype, R, x, static_cast<long long>(n), y, workspace,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

QR_EXPORT size_t qr_fc_tile_bytes(int bits) { return fc_bits_ok(bits) ? size_t(256) * size_t(bits) + 128 : 0; }

QR_EXPORT size_t qr_fc_wire_bytes(int bits, size_t n) { return fc_wire_bytes(bits, n); }

QR_EXPORT qr_status_t qr_fc_encode(int bits, qr_dtype_t dtype, const void *x, size_t n, void *wire,
                                   qr_stream_t stream) {
    if (!x || !wire || n == 0) return QR_ERR_INVALID_ARG;
    if (!fc_bits_ok(bits) || !dtype_ok(dtype)) return QR_ERR_UNSUPPORTED;
    const size_t W = fc_wire_bytes(bits, n);
    if (!value_bytes_ok(n) || W == 0) return QR_ERR_SIZE;
    if (!aligned16(x) || !aligned16(wire)) return QR_ERR_MISALIGNED;
    if (overlaps(wire, W, x, 2 * n)) return QR_ERR_INVALID_ARG;
    return from_cuda(qrk::launch_fc_encode(bits, dtype, x, static_cast<long long>(n), wire,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

QR_EXPORT qr_status_t qr_fc_decode(int bits, qr_dtype_t dtype, const void *wire, size_t n, void *y,
                                   qr_stream_t stream) {
    if (!wire || !y || n == 0) return QR_ERR_INVALID_ARG;
    if (!fc_bits_ok(bits) || !dtype_ok(dtype)) return QR_ERR_UNSUPPORTED;
    const size_t W = fc_wire_bytes(bits, n);
    if (!value_bytes_ok(n) || W == 0) return QR_ERR_SIZE;
    if (!aligned16(wire) || !aligned16(y)) return QR_ERR_MISALIGNED;
    if (overlaps(y, 2 * n, wire, W)) return QR_ERR_INVALID_ARG;
    return from_cuda(qrk::launch_fc_decode(bits, dtype, wire, static_cast<long long>(n), y,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

namespace {

qr_status_t fc_segment_reduce_common(int bits_in, int bits_out, int R, const void *const *wires, size_t n,
                                     void *out_wire, int ctas, bool staged, qr_stream_t stream) {
    if (!wires || !out_wire || n == 0 || R < 1 || ctas < 0) return QR_ERR_INVALID_ARG;
    for (int r = 0; r < R && r < QR_MAX_RANKS; ++r)
        if (!wires[r]) return QR_ERR_INVALID_ARG;
    if (!fc_pair_ok(bits_in, bits_out) || R > QR_MAX_RANKS) return QR_ERR_UNSUPPORTED;
    const size_t Wi = fc_wire_bytes(bits_in, n), Wo = fc_wire_bytes(bits_out, n);
    if (!value_bytes_ok(n) || Wi == 0 || Wo == 0) return QR_ERR_SIZE;
    if (!aligned16(out_wire)) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r)
        if (!aligned16(wires[r])) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r) {
        // in place only when the widths match (the tiles then line up)
        if (bits_in == bits_out ? bad_alias(out_wire, Wo, wires[r], Wi) : overlaps(out_wire, Wo, wires[r], Wi))
            return QR_ERR_INVALID_ARG;
    }
    if (staged)
        return from_cuda(qrk::launch_fc_reduce_staged(bits_in, bits_out, R, wires, static_cast<long long>(n), out_wire,
                                                      ctas, reinterpret_cast<cudaStream_t>(stream)));
    return from_cuda(qrk::launch_fc_reduce(bits_in, bits_out, R, wires, static_cast<long long>(n), out_wire,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

QR_EXPORT qr_status_t qr_fc_segment_reduce(int bits_in, int bits_out, int R, const void *const *wires, size_t n,
                                           void *out_wire, qr_stream_t stream) {
    return fc_segment_reduce_common(bits_in, bits_out, R, wires, n, out_wire, 0, false, stream);
}

QR_EXPORT qr_status_t qr_fc_segment_reduce_staged(int bits_in, int bits_out, int R, const void *const *wires,
                                                  size_t n, void *out_wire, int ctas, qr_stream_t stream) {
    return fc_segment_reduce_common(bits_in, bits_out, R, wires, n, out_wire, ctas, true, stream);
}

namespace {

qr_status_t fc_allreduce_common(int bits_rs, int bits_ag, qr_dtype_t dtype, int R, const void *const *x, size_t n,
                                void *y, int ctas, bool staged, qr_stream_t stream) {
    if (!x || !y || n == 0 || R < 1 || ctas < 0) return QR_ERR_INVALID_ARG;
    for (int r = 0; r < R && r < QR_MAX_RANKS; ++r)
        if (!x[r]) return QR_ERR_INVALID_ARG;
    if (!fc_pair_ok(bits_rs, bits_ag) || !dtype_ok(dtype) || R > QR_MAX_RANKS) return QR_ERR_UNSUPPORTED;
    if (!value_bytes_ok(n) || fc_wire_bytes(bits_rs, n) == 0) return QR_ERR_SIZE;
    const size_t V = 2 * n;
    if (!aligned16(y)) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r)
        if (!aligned16(x[r])) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r)
        if (bad_alias(y, V, x[r], V)) return QR_ERR_INVALID_ARG;
    if (staged) {
        const auto a32 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; };
        if (!a32(y)) return QR_ERR_MISALIGNED;
        for (int r = 0; r < R; ++r)
            if (!a32(x[r])) return QR_ERR_MISALIGNED;
        return from_cuda(qrk::launch_fc_allreduce_staged(bits_rs, bits_ag, dtype, R, x, static_cast<long long>(n), y,
                                                         ctas, reinterpret_cast<cudaStream_t>(stream)));
    }
    return from_cuda(qrk::launch_fc_allreduce(bits_rs, bits_ag, dtype, R, x, static_cast<long long>(n), y, ctas,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

QR_EXPORT qr_status_t qr_fc_allreduce(int bits_rs, int bits_ag, qr_dtype_t dtype, int R, const void *const *x,
                                      size_t n, void *y, qr_stream_t stream) {
    return fc_allreduce_common(bits_rs, bits_ag, dtype, R, x, n, y, 0, false, stream);
}

QR_EXPORT qr_status_t qr_fc_allreduce_ctas(int bits_rs, int bits_ag, qr_dtype_t dtype, int R, const void *const *x,
                                           size_t n, void *y, int ctas, qr_stream_t stream) {
    return fc_allreduce_common(bits_rs, bits_ag, dtype, R, x, n, y, ctas, false, stream);
}

QR_EXPORT qr_status_t qr_fc_allreduce_staged(int bits_rs, int bits_ag, qr_dtype_t dtype, int R, const void *const *x,
                                             size_t n, void *y, int ctas, qr_stream_t stream) {
    return fc_allreduce_common(bits_rs, bits_ag, dtype, R, x, n, y, ctas, true, stream);
}

QR_EXPORT const char *qr_status_string(qr_status_t status) {
    switch (status) {
        case QR_OK: return "QR_OK";
        case QR_ERR_INVALID_ARG: return "QR_ERR_INVALID_ARG: null pointer, zero size, R < 1 or partial aliasing";
        case QR_ERR_UNSUPPORTED: return "QR_ERR_UNSUPPORTED: bits not in {3,4,6,8}, unknown dtype or R > 8";
        case QR_ERR_MISALIGNED: return "QR_ERR_MISALIGNED: a device pointer is not 16-byte aligned";
        case QR_ERR_SIZE: return "QR_ERR_SIZE: a byte count overflows size_t";
        case QR_ERR_CUDA: return "QR_ERR_CUDA: the CUDA runtime reported an error";
    }
    return "QR_ERR_UNKNOWN: not a qr_status_t value";
}

QR_EXPORT qr_status_t qr_encode(int bits, qr_dtype_t dtype, const void *x, size_t n, void *wire,
                                qr_stream_t stream) {
    if (!x || !wire || n == 0) return QR_ERR_INVALID_ARG;
    if (!bits_ok(bits) || !dtype_ok(dtype)) return QR_ERR_UNSUPPORTED;
    const size_t W = wire_bytes(bits, n);
    if (!value_bytes_ok(n) || W == 0) return QR_ERR_SIZE;
    if (!aligned16(x) || !aligned16(wire)) return QR_ERR_MISALIGNED;
    if (overlaps(wire, W, x, 2 * n)) return QR_ERR_INVALID_ARG;
    return from_cuda(qrk::launch_encode(bits, dtype, x, static_cast<long long>(n), wire,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

QR_EXPORT qr_status_t qr_decode(int bits, qr_dtype_t dtype, const void *wire, size_t n, void *y,
                                qr_stream_t stream) {
    if (!wire || !y || n == 0) return QR_ERR_INVALID_ARG;
    if (!bits_ok(bits) || !dtype_ok(dtype)) return QR_ERR_UNSUPPORTED;
    const size_t W = wire_bytes(bits, n);
    if (!value_bytes_ok(n) || W == 0) return QR_ERR_SIZE;
    if (!aligned16(wire) || !aligned16(y)) return QR_ERR_MISALIGNED;
    if (overlaps(y, 2 * n, wire, W)) return QR_ERR_INVALID_ARG;
    return from_cuda(qrk::launch_decode(bits, dtype, wire, static_cast<long long>(n), y,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

namespace {

qr_status_t segment_reduce_common(int bits, int R, const void *const *wires, size_t n, void *out_wire, int ctas,
                                  bool staged, qr_stream_t stream) {
    if (!wires || !out_wire || n == 0 || R < 1 || ctas < 0) return QR_ERR_INVALID_ARG;
    for (int r = 0; r < R && r < QR_MAX_RANKS; ++r)
        if (!wires[r]) return QR_ERR_INVALID_ARG;
    if (!bits_ok(bits) || R > QR_MAX_RANKS) return QR_ERR_UNSUPPORTED;
    const size_t W = wire_bytes(bits, n);
    if (!value_bytes_ok(n) || W == 0) return QR_ERR_SIZE;
    if (!aligned16(out_wire)) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r)
        if (!aligned16(wires[r])) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r)
        if (bad_alias(out_wire, W, wires[r], W)) return QR_ERR_INVALID_ARG;
    if (staged)
        return from_cuda(qrk::launch_reduce_staged(bits, R, wires, static_cast<long long>(n), out_wire, ctas,
                                                   reinterpret_cast<cudaStream_t>(stream)));
    return from_cuda(qrk::launch_reduce(bits, R, wires, static_cast<long long>(n), out_wire,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

QR_EXPORT qr_status_t qr_segment_reduce(int bits, int R, const void *const *wires, size_t n,
                                        void *out_wire, qr_stream_t stream) {
    return segment_reduce_common(bits, R, wires, n, out_wire, 0, false, stream);
}

QR_EXPORT qr_status_t qr_segment_reduce_staged(int bits, int R, const void *const *wires, size_t n,
                                               void *out_wire, int ctas, qr_stream_t stream) {
    return segment_reduce_common(bits, R, wires, n, out_wire, ctas, true, stream);
}

namespace {

qr_status_t allreduce_common(int bits, qr_dtype_t dtype, int R, const void *const *x, size_t n, void *y,
                             void *const *wire_out, void *red_out, int ctas, qr_stream_t stream,
                             bool staged = false) {
    if (!x || !y || n == 0 || R < 1 || ctas < 0) return QR_ERR_INVALID_ARG;
    for (int r = 0; r < R && r < QR_MAX_RANKS; ++r) {
        if (!x[r]) return QR_ERR_INVALID_ARG;
        if (wire_out && !wire_out[r]) return QR_ERR_INVALID_ARG;
    }
    if (!bits_ok(bits) || !dtype_ok(dtype) || R > QR_MAX_RANKS) return QR_ERR_UNSUPPORTED;
    const size_t W = wire_bytes(bits, n);
    if (!value_bytes_ok(n) || W == 0) return QR_ERR_SIZE;
    const size_t V = 2 * n;
    if (!aligned16(y) || (red_out && !aligned16(red_out))) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r)
        if (!aligned16(x[r]) || (wire_out && !aligned16(wire_out[r]))) return QR_ERR_MISALIGNED;
    // outputs: y (may equal an input exactly), the R rank wires and the reduced wire
    for (int r = 0; r < R; ++r) {
        if (bad_alias(y, V, x[r], V)) return QR_ERR_INVALID_ARG;
        if (wire_out) {
            for (int i = 0; i < R; ++i)
                if (overlaps(wire_out[r], W, x[i], V)) return QR_ERR_INVALID_ARG;
            if (overlaps(wire_out[r], W, y, V)) return QR_ERR_INVALID_ARG;
            for (int i = 0; i < r; ++i)
                if (overlaps(wire_out[r], W, wire_out[i], W)) return QR_ERR_INVALID_ARG;
            if (red_out && overlaps(wire_out[r], W, red_out, W)) return QR_ERR_INVALID_ARG;
        }
        if (red_out && overlaps(red_out, W, x[r], V)) return QR_ERR_INVALID_ARG;
    }
    if (red_out && overlaps(red_out, W, y, V)) return QR_ERR_INVALID_ARG;
    if (staged) {
        const auto a32 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; };
        if (!a32(y)) return QR_ERR_MISALIGNED;
        for (int r = 0; r < R; ++r)
            if (!a32(x[r])) return QR_ERR_MISALIGNED;
        return from_cuda(qrk::launch_allreduce_staged(bits, dtype, R, x, static_cast<long long>(n), y, ctas,
                                                      reinterpret_cast<cudaStream_t>(stream)));
    }
    return from_cuda(qrk::launch_allreduce(bits, dtype, R, x, static_cast<long long>(n), y, wire_out, red_out,
                                           ctas, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

QR_EXPORT qr_status_t qr_allreduce(int bits, qr_dtype_t dtype, int R, const void *const *x, size_t n, void *y,
                                   qr_stream_t stream) {
    return allreduce_common(bits, dtype, R, x, n, y, nullptr, nullptr, 0, stream);
}

QR_EXPORT qr_status_t qr_allreduce_emit(int bits, qr_dtype_t dtype, int R, const void *const *x, size_t n,
                                        void *y, void *const *wire_out, void *red_out, qr_stream_t stream) {
    return allreduce_common(bits, dtype, R, x, n, y, wire_out, red_out, 0, stream);
}

QR_EXPORT qr_status_t qr_allreduce_staged(int bits, qr_dtype_t dtype, int R, const void *const *x, size_t n,
                                          void *y, int ctas, qr_stream_t stream) {
    return allreduce_common(bits, dtype, R, x, n, y, nullptr, nullptr, ctas, stream, true);
}

QR_EXPORT qr_status_t qr_allreduce_ctas(int bits, qr_dtype_t dtype, int R, const void *const *x, size_t n,
                                        void *y, int ctas, qr_stream_t stream) {
    return allreduce_common(bits, dtype, R, x, n, y, nullptr, nullptr, ctas, stream);
}

// ---------------------------------------------------------------------------
// the FP4 codec: the INT4 tile with E2M1 elements
// ---------------------------------------------------------------------------

QR_EXPORT size_t qr_fp4_tile_bytes(void) { return tile_bytes(4); }

QR_EXPORT size_t qr_fp4_wire_bytes(size_t n) { return wire_bytes(4, n); }

QR_EXPORT qr_status_t qr_fp4_encode(qr_dtype_t dtype, const void *x, size_t n, void *wire, qr_stream_t stream) {
    if (!x || !wire || n == 0) return QR_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return QR_ERR_UNSUPPORTED;
    const size_t W = wire_bytes(4, n);
    if (!value_bytes_ok(n) || W == 0) return QR_ERR_SIZE;
    if (!aligned16(x) || !aligned16(wire)) return QR_ERR_MISALIGNED;
    if (overlaps(wire, W, x, 2 * n)) return QR_ERR_INVALID_ARG;
    return from_cuda(qrk::launch_fp4_encode(dtype, x, static_cast<long long>(n), wire,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

QR_EXPORT qr_status_t qr_fp4_decode(qr_dtype_t dtype, const void *wire, size_t n, void *y, qr_stream_t stream) {
    if (!wire || !y || n == 0) return QR_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return QR_ERR_UNSUPPORTED;
    const size_t W = wire_bytes(4, n);
    if (!value_bytes_ok(n) || W == 0) return QR_ERR_SIZE;
    if (!aligned16(wire) || !aligned16(y)) return QR_ERR_MISALIGNED;
    if (overlaps(y, 2 * n, wire, W)) return QR_ERR_INVALID_ARG;
    return from_cuda(qrk::launch_fp4_decode(dtype, wire, static_cast<long long>(n), y,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

QR_EXPORT qr_status_t qr_fp4_segment_reduce(int R, const void *const *wires, size_t n, void *out_wire, int ctas,
                                            qr_stream_t stream) {
    if (!wires || !out_wire || n == 0 || R < 1 || ctas < 0) return QR_ERR_INVALID_ARG;
    for (int r = 0; r < R && r < QR_MAX_RANKS; ++r)
        if (!wires[r]) return QR_ERR_INVALID_ARG;
    if (R > QR_MAX_RANKS) return QR_ERR_UNSUPPORTED;
    const size_t W = wire_bytes(4, n);
    if (!value_bytes_ok(n) || W == 0) return QR_ERR_SIZE;
    if (!aligned16(out_wire)) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r)
        if (!aligned16(wires[r])) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r)
        if (bad_alias(out_wire, W, wires[r], W)) return QR_ERR_INVALID_ARG;
    return from_cuda(qrk::launch_fp4_reduce(R, wires, static_cast<long long>(n), out_wire, ctas,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

QR_EXPORT qr_status_t qr_fp4_allreduce(qr_dtype_t dtype, int R, const void *const *x, size_t n, void *y, int ctas,
                                       qr_stream_t stream) {
    if (!x || !y || n == 0 || R < 1 || ctas < 0) return QR_ERR_INVALID_ARG;
    for (int r = 0; r < R && r < QR_MAX_RANKS; ++r)
        if (!x[r]) return QR_ERR_INVALID_ARG;
    if (!dtype_ok(dtype) || R > QR_MAX_RANKS) return QR_ERR_UNSUPPORTED;
    if (!value_bytes_ok(n) || wire_bytes(4, n) == 0) return QR_ERR_SIZE;
    const auto a32 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; };
    if (!a32(y)) return QR_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r)
        if (!a32(x[r])) return QR_ERR_MISALIGNED;
    const size_t V = 2 * n;
    for (int r = 0; r < R; ++r)
        if (bad_alias(y, V, x[r], V)) return QR_ERR_INVALID_ARG;
    return from_cuda(qrk::launch_fp4_allreduce(dtype, R, x, static_cast<long long>(n), y, ctas,
                                               reinterpret_cast<cudaStream_t>(stream)));
}
