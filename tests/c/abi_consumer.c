/* A plain C11 consumer of the library's C ABI: compiled and run by the host tests (no GPU
 * calls): the header must be valid C, and the host-side checks must answer as documented. */
#include <stdio.h>

#include "spl.h"
#include "spl_checked.h" /* declarations only: the reader is exported by the checked build */

static int fails = 0;

static void expect(int cond, const char* what) {
    if (!cond) {
        printf("FAIL: %s\n", what);
        ++fails;
    }
}

int main(void) {
    spl_codec v = {2048u, 32u, SPL_SCALE_MEAN_ABS};
    spl_codec bad = {1024u, 16u, SPL_SCALE_MAX_ABS};
    spl_tensor t = {0, 0, 0};
    expect(spl_num_chunks(4097) == 2, "spl_num_chunks");
    expect(spl_codec_record_bytes(0) == SPL_RECORD_BYTES, "default record bytes");
    expect(spl_codec_record_bytes(&v) == 52, "variant record bytes");
    expect(spl_codec_record_bytes(&bad) == -1, "unsupported codec");
    expect(spl_codec_num_chunks(&v, 2049) == 2, "variant chunk count");
    expect(spl_status_string(SPL_ERR_ALIGNMENT)[0] != '\0', "status string");
    expect(spl_last_cuda_error() == 0, "no CUDA error yet");
    /* argument errors are answered on the host before any CUDA call */
    expect(spl_ef_compress(0, SPL_F32, 0, 0, 1.0f, 0, 0, 0, 0) == SPL_OK, "empty compress");
    expect(spl_ef_compress_multi(&t, 0, SPL_F32, 1.0f, 0, 0, 0, 0) == SPL_ERR_INVALID_ARG,
           "empty table");
    expect(spl_ef_compress_codec(&bad, &t, 1, SPL_F32, 1.0f, 0, 0, 0, 0) == SPL_ERR_INVALID_ARG,
           "unsupported codec rejected");
    expect(spl_decode_aggregate(0, 0, 0, 16, 0, 0, 0.0f, 1, 0, 0) == SPL_ERR_INVALID_ARG,
           "P = 0 rejected");
    expect(spl_decode_aggregate(0, 0, SPL_P_MAX + 1, 16, 0, 0, 0.0f, 0, 0, 0) ==
               SPL_ERR_INVALID_ARG, "P above SPL_P_MAX rejected");
    expect(SPL_PAYLOAD_BYTES == SPL_RECORD_BYTES && SPL_P_MAX == SPL_MAX_PEERS, "aliases");
    /* a flags word read back maps to a status, most severe first */
    expect(spl_flags_status(0u) == SPL_OK, "no flags");
    expect(spl_flags_status(SPL_FLAG_NONFINITE) == SPL_ERR_NONFINITE, "non-finite");
    expect(spl_flags_status(SPL_FLAG_BAD_RECORD | SPL_FLAG_NONFINITE) == SPL_ERR_BAD_PAYLOAD,
           "bad record before non-finite");
    expect(spl_flags_status(SPL_FLAG_TIMEOUT | SPL_FLAG_BAD_RECORD) == SPL_ERR_TIMEOUT,
           "timeout first");
    expect(spl_flags_status(SPL_FLAG_COPY_PENDING) == SPL_ERR_TIMEOUT, "copy pending");
    expect(spl_status_string(SPL_ERR_BAD_PAYLOAD)[0] != 'u', "status string of a flag status");
    expect(spl_pack(0, 0, 0, 0, 0) == SPL_OK, "empty pack");
    expect(SPL_DEBUG_WORDS == 16 && SPL_DEBUG_GENERIC < SPL_DEBUG_WORDS, "debug word layout");
    if (fails == 0) printf("ok\n");
    return fails != 0;
}
