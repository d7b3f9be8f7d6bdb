/*
 * qr_c_client.c -- a plain C11 caller of libqr.so (no C++, no Python, no
 * torch): the boundary used as include/qr.h states it.  It checks, on the
 * current CUDA device, for R = 4 ranks of n bf16 values (a ragged tail) and
 * every code width:
 *   - the fused all-reduce, the unfused steps (encode, Phase-1B, decode) and
 *     the two-shot exchange give the same bytes;
 *   - every wire, the reduced wire and the output equal the C oracle's
 *     (oracle/qr_oracle.h, test infrastructure), byte for byte;
 *   - the per-rank two-shot calls of every codec (symmetric INT4, the
 *     asymmetric 4->8 pair, FP4), each rank's send, then each owner's
 *     reduce, then each rank's decode into R workspaces of this process:
 *     every rank's output equals the oracle's all-reduce;
 *   - bad arguments return their status codes without launching anything;
 *   - no device-side wait ran out.
 * Exit status 0 and the line "qr_c_client ok" on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "qr.h"
#include "qr_oracle.h"

#define R 4

static int failures = 0;

#define CUDA_OK(call)                                                                          \
    do {                                                                                       \
        cudaError_t e_ = (call);                                                               \
        if (e_ != cudaSuccess) {                                                               \
            fprintf(stderr, "%s:%d: %s: %s\n", __FILE__, __LINE__, #call, cudaGetErrorString(e_)); \
            exit(2);                                                                           \
        }                                                                                      \
    } while (0)

static void expect(int cond, const char *what) {
    if (!cond) {
        fprintf(stderr, "FAILED: %s\n", what);
        ++failures;
    }
}

static uint32_t lcg(uint32_t *s) {
    *s = *s * 1664525u + 1013904223u;
    return *s;
}

/* The per-rank calls of one codec (0: symmetric INT4, 1: asymmetric 4->8,
 * 2: FP4) for all R ranks from this process; every rank's output is compared
 * with `ref`. */
static void per_rank(int codec, void *const *dx, size_t n, void *const *dys, const uint16_t *ref, uint16_t *host) {
    const size_t need = codec == 0   ? qr_twoshot_peer_workspace_bytes(4, R, n)
                        : codec == 1 ? qr_fc_twoshot_peer_workspace_bytes(4, 8, R, n)
                                     : qr_fp4_twoshot_peer_workspace_bytes(R, n);
    expect(need > 0, "peer workspace bytes");
    void *ws[R];
    for (int r = 0; r < R; ++r) CUDA_OK(cudaMalloc(&ws[r], need));
    for (int j = 0; j < R; ++j) {
        const qr_status_t st = codec == 0   ? qr_twoshot_peer_send(4, QR_BF16, R, j, dx[j], n, ws, NULL)
                               : codec == 1 ? qr_fc_twoshot_peer_send(4, 8, QR_BF16, R, j, dx[j], n, ws, NULL)
                                            : qr_fp4_twoshot_peer_send(QR_BF16, R, j, dx[j], n, ws, NULL);
        expect(st == QR_OK, "per-rank send");
    }
    for (int j = 0; j < R; ++j) {
        const qr_status_t st = codec == 0   ? qr_twoshot_peer_reduce(4, R, j, n, ws, NULL)
                               : codec == 1 ? qr_fc_twoshot_peer_reduce(4, 8, R, j, n, ws, NULL)
                                            : qr_fp4_twoshot_peer_reduce(R, j, n, ws, NULL);
        expect(st == QR_OK, "per-rank reduce");
    }
    for (int j = 0; j < R; ++j) {
        const qr_status_t st = codec == 0   ? qr_twoshot_peer_decode(4, QR_BF16, R, n, ws[j], dys[j], NULL)
                               : codec == 1 ? qr_fc_twoshot_peer_decode(4, 8, QR_BF16, R, n, ws[j], dys[j], NULL)
                                            : qr_fp4_twoshot_peer_decode(QR_BF16, R, n, ws[j], dys[j], NULL);
        expect(st == QR_OK, "per-rank decode");
    }
    expect(qr_twoshot_peer_send(4, QR_BF16, R, R, dx[0], n, ws, NULL) == QR_ERR_INVALID_ARG, "rank out of range");
    expect(qr_fc_twoshot_peer_reduce(8, 4, R, 0, n, ws, NULL) == QR_ERR_UNSUPPORTED, "width pair 8->4");
    CUDA_OK(cudaDeviceSynchronize());
    for (int j = 0; j < R; ++j) {
        CUDA_OK(cudaMemcpy(host, dys[j], n * 2, cudaMemcpyDeviceToHost));
        expect(memcmp(host, ref, n * 2) == 0, "per-rank output equals the oracle's");
    }
    for (int r = 0; r < R; ++r) CUDA_OK(cudaFree(ws[r]));
}

int main(void) {
    const size_t n = 2048 * 37 + 11;
    uint32_t seed = 12345u;
    uint16_t *hx[R];
    void *dx[R];
    for (int r = 0; r < R; ++r) {
        hx[r] = (uint16_t *)malloc(n * 2);
        for (size_t i = 0; i < n; ++i) {
            float v = ((float)(lcg(&seed) >> 8) * (1.0f / 16777216.0f) * 8.0f - 4.0f) * (float)(1 + r);
            if (i % 997 == 0) v *= 50.0f;
            hx[r][i] = orc_f32_to_bf16(v);
        }
        CUDA_OK(cudaMalloc(&dx[r], n * 2));
        CUDA_OK(cudaMemcpy(dx[r], hx[r], n * 2, cudaMemcpyHostToDevice));
    }
    void *dy, *dy2, *dys[R];
    CUDA_OK(cudaMalloc(&dy, n * 2));
    CUDA_OK(cudaMalloc(&dy2, n * 2));
    for (int r = 0; r < R; ++r) CUDA_OK(cudaMalloc(&dys[r], n * 2));
    uint16_t *hy = (uint16_t *)malloc(n * 2), *hy2 = (uint16_t *)malloc(n * 2), *href = (uint16_t *)malloc(n * 2);

    const int widths[4] = {8, 6, 4, 3};
    for (int wi = 0; wi < 4; ++wi) {
        const int bits = widths[wi];
        const size_t W = qr_wire_bytes(bits, n);
        void *dw[R], *dred;
        for (int r = 0; r < R; ++r) CUDA_OK(cudaMalloc(&dw[r], W));
        CUDA_OK(cudaMalloc(&dred, W));
        const size_t ws_bytes = qr_twoshot_workspace_bytes(bits, R, n);
        void *dws;
        CUDA_OK(cudaMalloc(&dws, ws_bytes));

        expect(qr_allreduce(bits, QR_BF16, R, (const void *const *)dx, n, dy, NULL) == QR_OK, "qr_allreduce");
        for (int r = 0; r < R; ++r) expect(qr_encode(bits, QR_BF16, dx[r], n, dw[r], NULL) == QR_OK, "qr_encode");
        expect(qr_segment_reduce(bits, R, (const void *const *)dw, n, dred, NULL) == QR_OK, "qr_segment_reduce");
        expect(qr_decode(bits, QR_BF16, dred, n, dy2, NULL) == QR_OK, "qr_decode");
        expect(qr_allreduce_twoshot(bits, QR_BF16, R, (const void *const *)dx, n, (void *const *)dys, dws, ws_bytes,
                                    NULL) == QR_OK,
               "qr_allreduce_twoshot");
        CUDA_OK(cudaDeviceSynchronize());

        /* the oracle, step by step */
        uint8_t *wref[R], *wgot = (uint8_t *)malloc(W), *redref = (uint8_t *)malloc(W);
        for (int r = 0; r < R; ++r) {
            wref[r] = (uint8_t *)malloc(W);
            expect(orc_encode(bits, 1, hx[r], n, wref[r]) == 0, "orc_encode");
            CUDA_OK(cudaMemcpy(wgot, dw[r], W, cudaMemcpyDeviceToHost));
            expect(memcmp(wgot, wref[r], W) == 0, "wire equals the oracle's");
        }
        expect(orc_segment_reduce(bits, R, (const uint8_t *const *)wref, n, redref) == 0, "orc_segment_reduce");
        CUDA_OK(cudaMemcpy(wgot, dred, W, cudaMemcpyDeviceToHost));
        expect(memcmp(wgot, redref, W) == 0, "reduced wire equals the oracle's");
        expect(orc_allreduce(bits, 1, R, (const uint16_t *const *)hx, n, href) == 0, "orc_allreduce");
        CUDA_OK(cudaMemcpy(hy, dy, n * 2, cudaMemcpyDeviceToHost));
        CUDA_OK(cudaMemcpy(hy2, dy2, n * 2, cudaMemcpyDeviceToHost));
        expect(memcmp(hy, href, n * 2) == 0, "fused output equals the oracle's");
        expect(memcmp(hy2, href, n * 2) == 0, "unfused output equals the oracle's");
        for (int r = 0; r < R; ++r) {
            CUDA_OK(cudaMemcpy(hy2, dys[r], n * 2, cudaMemcpyDeviceToHost));
            expect(memcmp(hy2, href, n * 2) == 0, "two-shot output equals the oracle's");
        }
        for (int r = 0; r < R; ++r) {
            free(wref[r]);
            CUDA_OK(cudaFree(dw[r]));
        }
        free(wgot);
        free(redref);
        CUDA_OK(cudaFree(dred));
        CUDA_OK(cudaFree(dws));
        printf("INT%d: fused, unfused and two-shot equal the oracle\n", bits);
    }

    /* the per-rank two-shot of each codec */
    static const char *const codec_names[3] = {"symmetric INT4", "asymmetric 4->8", "FP4"};
    for (int codec = 0; codec < 3; ++codec) {
        const int rc = codec == 0   ? orc_allreduce(4, 1, R, (const uint16_t *const *)hx, n, href)
                       : codec == 1 ? orc_fc_allreduce(4, 8, 1, R, (const uint16_t *const *)hx, n, href)
                                    : orc_fp4_allreduce(1, R, (const uint16_t *const *)hx, n, href);
        expect(rc == 0, "oracle all-reduce");
        per_rank(codec, dx, n, dys, href, hy);
        printf("%s: the per-rank two-shot equals the oracle on every rank\n", codec_names[codec]);
    }

    /* bad arguments: status codes, nothing launched */
    expect(qr_allreduce(5, QR_BF16, R, (const void *const *)dx, n, dy, NULL) == QR_ERR_UNSUPPORTED, "bits 5");
    expect(qr_allreduce(4, QR_BF16, 0, (const void *const *)dx, n, dy, NULL) == QR_ERR_INVALID_ARG, "R = 0");
    expect(qr_allreduce(4, QR_BF16, R, (const void *const *)dx, 0, dy, NULL) == QR_ERR_INVALID_ARG, "n = 0");
    expect(qr_allreduce(4, QR_BF16, R, (const void *const *)dx, n, NULL, NULL) == QR_ERR_INVALID_ARG, "y = NULL");
    expect(qr_allreduce(4, QR_BF16, R, (const void *const *)dx, n, (char *)dy + 2, NULL) == QR_ERR_MISALIGNED,
           "misaligned y");
    expect(qr_status_string(QR_ERR_SIZE) != NULL, "status string");

    unsigned timeouts = 1;
    expect(qr_wait_timeouts(&timeouts) == QR_OK && timeouts == 0, "no device-side wait ran out");

    for (int r = 0; r < R; ++r) {
        free(hx[r]);
        CUDA_OK(cudaFree(dx[r]));
        CUDA_OK(cudaFree(dys[r]));
    }
    CUDA_OK(cudaFree(dy));
    CUDA_OK(cudaFree(dy2));
    free(hy);
    free(hy2);
    free(href);
    if (failures) {
        fprintf(stderr, "qr_c_client: %d check(s) failed\n", failures);
        return 1;
    }
    printf("qr_c_client ok\n");
    return 0;
}
