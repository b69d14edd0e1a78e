"""The C-ABI library: it builds, loads, exports every declared entry point, and
validates arguments on the host.  No GPU needed (no compute calls)."""
import ctypes

import pytest

import lm_head_vocab_gb300._lib as L


@pytest.fixture(scope="module")
def lib():
    L.build()
    return L.load()


def test_exports_every_declared_symbol(lib):
    names = L.exported_names()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
        ctypes.cast(getattr(lib, n), ctypes.c_void_p)   # resolvable


def test_status_strings(lib):
    for s in range(8):
        assert L.lmloss_status_string(s) != "unknown status"
    assert L.lmloss_status_string(99) == "unknown status"


def _args(**kw):
    a = L.lmloss_args()
    a.logits = 0x10000
    a.T, a.V, a.ld = 4, 10, 16
    a.dtype = L.LMLOSS_BF16
    a.reduction = L.LMLOSS_REDUCE_TOKEN_MEAN
    a.targets = 0x20000
    a.loss_out = 0x30000
    a.ce_weight = 1.0
    a.temperature = 1.0
    a.denominator = 1.0
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,expect", [
    ({}, L.LMLOSS_OK),
    ({"V": 0}, L.LMLOSS_ERR_INVALID_ARG),
    ({"ld": 9}, L.LMLOSS_ERR_INVALID_ARG),
    ({"T": -1}, L.LMLOSS_ERR_INVALID_ARG),
    ({"dtype": 7}, L.LMLOSS_ERR_INVALID_ARG),
    ({"reduction": 3}, L.LMLOSS_ERR_INVALID_ARG),
    ({"loss_out": None}, L.LMLOSS_ERR_INVALID_ARG),
    ({"targets": None}, L.LMLOSS_ERR_INVALID_ARG),
    ({"logits": None}, L.LMLOSS_ERR_INVALID_ARG),
    ({"logits": None, "targets": None, "T": 0}, L.LMLOSS_OK),
    ({"logits": 0x10001}, L.LMLOSS_ERR_INVALID_ARG),                       # bf16 misaligned
    ({"dtype": L.LMLOSS_FP32, "logits": 0x10002}, L.LMLOSS_ERR_INVALID_ARG),
    ({"grad_out": 0x50008}, L.LMLOSS_ERR_INVALID_ARG),                     # phase differs mod 16
    ({"grad_out": 0x50000}, L.LMLOSS_OK),
    ({"grad_out": 0x10000}, L.LMLOSS_OK),                                   # in place
    ({"reduction": L.LMLOSS_REDUCE_SUM, "denominator": 0.0}, L.LMLOSS_ERR_INVALID_ARG),
    ({"reduction": L.LMLOSS_REDUCE_SUM, "denominator": 3.0}, L.LMLOSS_OK),
    ({"teacher_logits": 0x60000, "kl_weight": 0.5}, L.LMLOSS_OK),
    ({"teacher_logits": 0x60000, "temperature": 2.0}, L.LMLOSS_OK),
    ({"teacher_logits": 0x60000, "temperature": 0.25}, L.LMLOSS_OK),
    ({"teacher_logits": 0x60000, "temperature": 0.0}, L.LMLOSS_ERR_INVALID_ARG),
    ({"teacher_logits": 0x60000, "temperature": -1.0}, L.LMLOSS_ERR_INVALID_ARG),
    ({"teacher_logits": 0x60000, "temperature": float("inf")}, L.LMLOSS_ERR_INVALID_ARG),
    ({"teacher_logits": 0x60000, "temperature": float("nan")}, L.LMLOSS_ERR_INVALID_ARG),
    ({"temperature": 0.0}, L.LMLOSS_OK),                                    # ignored without a teacher
    ({"teacher_logits": 0x60004}, L.LMLOSS_ERR_INVALID_ARG),
    ({"segment_ids": 0x70000, "num_segments": 2, "advantages": 0x71000, "old_logprobs": 0x72000}, L.LMLOSS_OK),
    ({"segment_ids": 0x70000, "num_segments": 2, "old_logprobs": 0x72000}, L.LMLOSS_ERR_INVALID_ARG),
    ({"segment_ids": 0x70000, "num_segments": 2, "advantages": 0x71000}, L.LMLOSS_ERR_INVALID_ARG),
    ({"segment_ids": 0x70000, "num_segments": -1, "advantages": 0x71000, "old_logprobs": 0x72000},
     L.LMLOSS_ERR_INVALID_ARG),
    ({"segment_ids": 0x70000, "num_segments": 2, "advantages": 0x71000, "old_logprobs": 0x72000,
      "teacher_logits": 0x60000}, L.LMLOSS_OK),                                   # GSPO with a teacher
    ({"segment_ids": 0x70000, "num_segments": 2, "advantages": 0x71000, "old_logprobs": 0x72000,
      "clip_eps_low": -0.1}, L.LMLOSS_ERR_INVALID_ARG),
])
def test_host_validation(lib, kw, expect):
    assert L.lmloss_check_args(_args(**kw)) == expect


def test_null_args_and_handle(lib):
    assert lib.lmloss_check_args(None) == L.LMLOSS_ERR_INVALID_ARG
    assert lib.lmloss_forward_backward(None, ctypes.byref(_args()), None) == L.LMLOSS_ERR_INVALID_ARG
    assert lib.lmloss_destroy(None) == L.LMLOSS_ERR_INVALID_ARG
    assert lib.lmloss_get_device_error(None) == L.LMLOSS_ERR_INVALID_ARG
    assert lib.lmloss_set_launch_config(None, 0, 0, 0) == L.LMLOSS_ERR_INVALID_ARG
    assert lib.lmloss_forward_backward_host(None, ctypes.byref(_args()), None, None, 0, None) == \
        L.LMLOSS_ERR_INVALID_ARG


def test_struct_layout_matches_header():
    # the ctypes mirror must follow the header's field order
    import re
    txt = open(L.HEADER).read()
    body = txt[txt.index("typedef struct {", txt.index("lmloss_handle;")):txt.index("} lmloss_args;")]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"(\w+)\s*;", body)
    assert fields == [f for f, _ in L.lmloss_args._fields_]


def test_call_info_layout_matches_header():
    import re
    txt = open(L.HEADER).read()
    i = txt.index("} lmloss_call_info;")
    body = txt[txt.rindex("typedef struct {", 0, i):i]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"(\w+)\s*;", body)
    assert fields == [f for f, _ in L.lmloss_call_info._fields_]
