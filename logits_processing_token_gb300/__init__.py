"""GB300-native per-step token selection: logits processors, greedy/multinomial
selection and assisted-generation verify, as CUDA kernels for sm_103a behind
the C ABI of include/tg.h.  This package is the thin Python binding."""
from .tg import (  # noqa: F401
    EXPORTS, TG_DTYPE_BF16, TG_DTYPE_F32, TG_ERR_CUDA, TG_ERR_INVALID_ARGUMENT, TG_ERR_OUT_OF_MEMORY,
    TG_ERR_UNSUPPORTED, TG_FLAG_BAD_ROW, TG_FLAG_BAD_STATE, TG_FLAG_HISTORY_ID_OUT_OF_RANGE, TG_FLAG_SLOW_PATH,
    TG_FLAG_TIMEOUT,
    TG_GREEDY, TG_MAX_PROCESSORS, TG_MAX_STATE_COLS, TG_MAX_VOCAB, TG_NOALLOC_MAX_BATCH, TG_OK, TG_PROC_BIAS,
    TG_PROC_SET, TG_SAMPLE, Config, TGError, load_library, make_params, tg_clear_status, tg_beam_keep, tg_beam_step,
    tg_next_num_candidates, tg_params, tg_process, tg_process_state, tg_query_status, tg_select, tg_select_state,
    tg_set_wait_limit, tg_status_string, tg_status_word, tg_verify, tg_verify_history,
)
