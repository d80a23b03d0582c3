"""ctypes mirrors of include/pcd.h: structures and function signatures."""
import ctypes

c_int, c_int32, c_int64, c_float, c_void_p, c_char_p = (ctypes.c_int, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                                       ctypes.c_void_p, ctypes.c_char_p)
P = ctypes.POINTER


class pcd_model_config(ctypes.Structure):
    _fields_ = [("n_layers", c_int), ("d_model", c_int), ("n_q_heads", c_int), ("n_kv_heads", c_int),
                ("head_dim", c_int), ("d_ff", c_int), ("vocab", c_int), ("rms_eps", c_float),
                ("rope_theta", c_float), ("tied_embedding", c_int), ("max_positions", c_int)]


class pcd_field(ctypes.Structure):
    _fields_ = [("scaffold", P(c_int32)), ("n_scaffold", c_int), ("cand_tokens", P(c_int32)),
                ("cand_offsets", P(c_int32)), ("n_cands", c_int), ("temperature", c_float),
                ("scoring", c_int), ("cand_label", P(c_int32)), ("n_labels", c_int)]


class pcd_field_result(ctypes.Structure):
    _fields_ = [("probs", P(c_float)), ("logprobs", P(c_float)), ("label", c_int32), ("mass", c_float),
                ("log_mass", c_float), ("margin", c_float), ("first_mass", c_float)]


class pcd_stats(ctypes.Structure):
    _fields_ = [("prefill_ms", c_float), ("compile_ms", c_float), ("branch_ms", c_float), ("readout_ms", c_float),
                ("total_ms", c_float), ("forward_passes", c_int), ("branch_tokens", c_int), ("readout_rows", c_int),
                ("h2d_bytes", c_int64), ("d2h_bytes", c_int64)]


# (name, restype, argtypes) of every entry point declared in include/*.h
SIGNATURES = [
    ("pcd_load_weights", c_int, [P(pcd_model_config), c_char_p, c_void_p, P(c_void_p)]),
    ("pcd_load_weights_host", c_int, [P(pcd_model_config), P(c_void_p), c_int, c_void_p, P(c_void_p)]),
    ("pcd_model_free", None, [c_void_p]),
    ("pcd_kv_bytes_per_token", c_int64, [c_void_p]),
    ("pcd_prefill", c_int, [c_void_p, P(c_int32), c_int, P(c_void_p)]),
    ("pcd_prefill_device", c_int, [c_void_p, c_void_p, c_int, P(c_void_p)]),
    ("pcd_prefill_extend", c_int, [c_void_p, c_void_p, P(c_int32), c_int, P(c_void_p)]),
    ("pcd_cache_length", c_int, [c_void_p]),
    ("pcd_cache_free", None, [c_void_p]),
    ("pcd_score", c_int, [c_void_p, c_void_p, P(pcd_field), c_int, P(pcd_field_result), P(pcd_stats)]),
    ("pcd_score_batch", c_int, [c_void_p, P(c_void_p), P(P(pcd_field)), P(c_int), c_int,
                                P(P(pcd_field_result)), P(pcd_stats)]),
    ("pcd_plan_create", c_int, [c_void_p, P(pcd_field), c_int, P(c_void_p)]),
    ("pcd_plan_free", None, [c_void_p]),
    ("pcd_plan_result_floats", c_int, [c_void_p]),
    ("pcd_score_plan_device", c_int, [c_void_p, c_void_p, c_void_p, c_void_p]),
    ("pcd_prefill_score", c_int, [c_void_p, P(c_int32), c_int, P(pcd_field), c_int, P(pcd_field_result),
                                  P(pcd_stats), P(c_void_p)]),
    ("pcd_prefill_score_plan_device", c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p, P(c_void_p)]),
    ("pcd_score_first_field_first", c_int, [c_void_p, c_void_p, P(pcd_field), c_int, P(c_int32), c_int,
                                            P(pcd_field_result), P(pcd_stats), P(c_void_p)]),
    ("pcd_prefill_score_first_field_first", c_int, [c_void_p, P(c_int32), c_int, P(pcd_field), c_int, P(c_int32),
                                                    c_int, P(pcd_field_result), P(pcd_stats), P(c_void_p)]),
    ("pcd_sync", c_int, [c_void_p]),
    ("pcd_profile_enable", c_int, [c_void_p, c_int]),
    ("pcd_profile_read", c_int, [c_void_p, P(c_int), P(c_float)]),
    ("pcd_abi_layout", c_int, [P(c_int32), c_int]),
    ("pcd_strerror", c_char_p, [c_int]),
    ("pcd_last_error", c_char_p, []),
    ("pcd_k_gemm_split", c_int, [c_void_p, c_void_p, c_int, c_int, c_void_p, c_int, c_int, c_int, c_int, c_void_p,
                                 c_int, c_int, c_int, c_void_p, c_void_p]),
    ("pcd_k_readout_scratch_bytes", c_int64, [c_int, c_int, c_int]),
    ("pcd_k_readout", c_int, [c_void_p, c_int, c_void_p, c_int, c_int, P(c_int32), P(c_int32), c_int, c_void_p,
                              c_void_p, c_void_p, c_int64, c_void_p, c_void_p]),
    ("pcd_k_readout_noalloc", c_int, [c_void_p, c_int, c_void_p, c_int, c_int, P(c_int32), P(c_int32), c_int,
                                      c_void_p, c_void_p, c_void_p, c_void_p]),
    ("pcd_plan_inspect", c_int, [c_void_p, c_int, c_int, P(c_int32), P(P(c_int32)), P(c_int32), c_int]),
    ("pcd_answer_line", c_int, [c_void_p, c_int, P(c_int32), c_int, P(c_int32), c_int]),
    ("pcd_k_gemm", c_int, [c_void_p, c_int, c_int, c_void_p, c_int, c_int, c_int, c_int, c_void_p, c_int,
                           c_int, c_int, c_int, c_void_p, c_void_p]),
    ("pcd_k_wait_probe", c_int, [c_int64, c_void_p, c_void_p, c_void_p]),
    ("pcd_k_gemm_swap", c_int, [c_void_p, c_void_p, c_int, c_int, c_void_p, c_int, c_int, c_int, c_int, c_void_p,
                                c_int, c_int, c_void_p, c_void_p]),
]


def declare(lib, sig):
    for name, res, args in SIGNATURES:
        sig(lib, name, res, args)
