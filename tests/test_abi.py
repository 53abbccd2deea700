"""The C-ABI library builds, loads without a GPU and exports every entry point
that include/ppo.h declares; host-side argument checks need no device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "ppo.h")).read()
    decl = r"^(?:ppo_status|const char \*)\s*(ppo_[a-z_0-9]+)\s*\("
    return sorted(set(re.findall(decl, src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from policy_rl_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 16
    for n in names:
        assert hasattr(lib, n), n


def test_binding_declares_the_same_symbols():
    from policy_rl_gb300 import _abi
    assert sorted(_abi.SYMBOLS) == _declared()


def test_host_side_argument_checks(lib):
    from policy_rl_gb300 import _abi, make_config
    L = _abi.load()
    assert L.ppo_status_string(2) == b"device pointer not 16-byte aligned"
    n = ctypes.c_int64()
    cfg = make_config(32, 64, 64, heads=(3, 2, 2), precision=0, max_batch=8192,
                      max_minibatch=2048)
    assert L.ppo_param_count(ctypes.byref(cfg), ctypes.byref(n)) == 0
    assert n.value == 64 * 32 + 64 + 64 * 64 + 64 + 8 * 64 + 8
    bad = make_config(32, 64, 64, heads=(30, 3), precision=0)   # C = 34 > 32
    assert L.ppo_param_count(ctypes.byref(bad), ctypes.byref(n)) == 4
    sz = ctypes.c_size_t()
    assert L.ppo_gae_workspace_bytes(0, 5, ctypes.byref(sz)) == 1
    assert L.ppo_gae_workspace_bytes(128, 64, ctypes.byref(sz)) == 0 and sz.value > 0
    assert L.ppo_perm_workspace_bytes(-1, ctypes.byref(sz)) == 1
    # misaligned device pointers are rejected before any CUDA call
    p = ctypes.c_void_p(0x1004)
    assert L.ppo_gae(p, p, p, p, 4, 4, 0.99, 0.95, p, p, None, None, None, 0, None) == 2
    assert L.ppo_minibatch_perm(0, 0, 16, p, p, 1 << 20, None) == 2


def test_recurrent_and_new_host_side_checks(lib):
    import oracle
    from policy_rl_gb300 import _abi, make_config, make_rnn_config
    L = _abi.load()
    n = ctypes.c_int64()
    # recurrent policy: the parameter count equals the oracle's layout
    for D, H, Ly, heads, G in ((3, 4, 2, (3, 2), 1), (64, 128, 4, (9, 2, 2, 2), 0)):
        cfg = make_rnn_config(D, H, Ly, heads, G)
        assert L.ppo_rnn_param_count(ctypes.byref(cfg), ctypes.byref(n)) == 0
        assert n.value == oracle.Rnn(D, H, Ly, heads, G).num_params
    assert L.ppo_rnn_param_count(ctypes.byref(make_rnn_config(3, 0, 2)), ctypes.byref(n)) == 1
    assert L.ppo_rnn_param_count(ctypes.byref(make_rnn_config(3, 512, 2)), ctypes.byref(n)) == 4
    assert L.ppo_rnn_param_count(ctypes.byref(make_rnn_config(3, 8, 9)), ctypes.byref(n)) == 4
    assert L.ppo_rnn_param_count(ctypes.byref(make_rnn_config(3, 8, 2, heads=(30, 3))),
                                 ctypes.byref(n)) == 4
    sz = ctypes.c_size_t()
    cfg = make_rnn_config(3, 4, 2, (3, 2), 1)
    assert L.ppo_rnn_workspace_bytes(ctypes.byref(cfg), 0, 2, ctypes.byref(sz)) == 1
    assert L.ppo_rnn_workspace_bytes(ctypes.byref(cfg), 6, 2, ctypes.byref(sz)) == 0
    assert sz.value > 0
    # invalid modes of the learner config
    bad = make_config(32, 64, 64, precision=0, adv_mode=3)
    assert L.ppo_param_count(ctypes.byref(bad), ctypes.byref(n)) == 1
    bad = make_config(32, 64, 64, precision=0, optimizer=2)
    assert L.ppo_param_count(ctypes.byref(bad), ctypes.byref(n)) == 1
    assert L.ppo_segment_advantage_workspace_bytes(ctypes.byref(sz)) == 0 and sz.value >= 16
