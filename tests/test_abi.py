"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports every
entry point include/kda.h declares, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_08_gb300 import binding
    if not os.path.exists(binding.LIB_PATH):
        from gated_delta_rule_08_gb300.build import build_library
        build_library()
    return binding.load_library()


def test_header_declares_the_entry_points():
    names = declared_functions()
    from gated_delta_rule_08_gb300 import binding
    assert set(binding.EXPORTS) <= set(names), names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libkda.so does not export {name}"


def test_only_the_api_is_exported(lib):
    out = os.popen(f"nm -D --defined-only {lib._name}").read()
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(declared_functions()), exported


def test_status_strings(lib):
    assert lib.kda_status_string(0) == b"KDA_OK"
    assert lib.kda_status_string(5) == b"KDA_ERR_WORKSPACE"


def test_workspace_size_host_logic(lib):
    f = lib.kda_chunk_fwd_workspace_size
    assert f(1, 8192, 32, 128, 128, 64, 0) > 0
    assert f(1, 8192, 32, 96, 128, 64, 0) == 0     # unsupported head dim
    assert f(1, 8192, 32, 128, 128, 32, 0) == 0    # only C = 64
    assert f(0, 8192, 32, 128, 128, 64, 0) == 0
    # grows with the chunk bound ceil(T/64) + B
    assert f(8, 8192, 32, 128, 128, 64, 1) > f(1, 8192, 32, 128, 128, 64, 1)


def test_bad_arguments_rejected_without_launch(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)
    # unsupported out dtype
    assert lib.kda_chunk_fwd(fake, fake, fake, fake, fake, None, None, fake, None, 1, 64, 1, 128, 128, 64, 0, 9,
                             None, fake, 1 << 20, None) == 2
    # unsupported chunk size / dims / dtype
    assert lib.kda_chunk_fwd(fake, fake, fake, fake, fake, None, None, fake, None, 1, 64, 1, 128, 128, 32, 0, 0,
                             None, fake, 1 << 20, None) == 2
    assert lib.kda_chunk_fwd(fake, fake, fake, fake, fake, None, None, fake, None, 1, 64, 1, 80, 128, 64, 0, 0,
                             None, fake, 1 << 20, None) == 2
    assert lib.kda_chunk_fwd(fake, fake, fake, fake, fake, None, None, fake, None, 1, 64, 1, 128, 128, 64, 7, 0,
                             None, fake, 1 << 20, None) == 2
    # null inputs, negative sizes
    assert lib.kda_chunk_fwd(None, fake, fake, fake, fake, None, None, fake, None, 1, 64, 1, 128, 128, 64, 0, 0,
                             None, fake, 1 << 20, None) == 1
    assert lib.kda_chunk_fwd(fake, fake, fake, fake, fake, None, None, fake, None, -1, 64, 1, 128, 128, 64, 0, 0,
                             None, fake, 1 << 20, None) == 1
    # out aliasing an input
    assert lib.kda_chunk_fwd(fake, fake, fake, fake, fake, None, None, fake, None, 1, 64, 1, 128, 128, 64, 0, 0,
                             None, fake, 1 << 20, None) == 1
    # workspace too small / misaligned
    other = P(0x2000)
    assert lib.kda_chunk_fwd(fake, fake, fake, fake, fake, None, None, other, None, 1, 64, 1, 128, 128, 64, 0, 0,
                             None, P(0x3000), 16, None) == 5
    assert lib.kda_chunk_fwd(fake, fake, fake, fake, fake, None, None, other, None, 1, 64, 1, 128, 128, 64, 0, 0,
                             None, P(0x3004), 1 << 30, None) == 5
    # decode
    assert lib.kda_decode_step(fake, fake, fake, fake, fake, fake, fake, fake, 4, 2, 128, 96, 8, 0, 0, None,
                               None) == 2
    assert lib.kda_decode_step(fake, fake, None, fake, fake, fake, fake, fake, 4, 2, 128, 128, 8, 0, 0, None,
                               None) == 1
    assert lib.kda_decode_step(fake, fake, fake, fake, fake, fake, fake, fake, -4, 2, 128, 128, 8, 0, 0, None,
                               None) == 1


def test_multi_token_and_checkpoint_arguments_rejected_without_launch(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)
    # decode_multi: negative token count, null values, unsupported dims
    assert lib.kda_decode_multi(fake, fake, fake, fake, fake, fake, fake, None, fake, 4, -1, 2, 128, 128, 8, 1, 0, 0,
                                None, None) == 1
    assert lib.kda_decode_multi(fake, fake, None, fake, fake, fake, fake, None, fake, 4, 3, 2, 128, 128, 8, 0, 0, 0,
                                None, None) == 1
    assert lib.kda_decode_multi(fake, fake, fake, fake, fake, fake, fake, None, fake, 4, 3, 2, 128, 96, 8, 0, 0, 0,
                                None, None) == 2
    # decode: v and the gate logits must be 16-byte aligned (the state pool too)
    odd = P(0x1008)
    assert lib.kda_decode_multi(fake, fake, odd, fake, fake, fake, fake, None, fake, 4, 3, 2, 128, 128, 8, 0, 0, 0,
                                None, None) == 1
    assert lib.kda_decode_step(fake, fake, odd, fake, fake, fake, fake, fake, 4, 2, 128, 128, 8, 0, 0, None,
                               None) == 1
    assert lib.kda_decode_step(fake, fake, fake, fake, fake, odd, fake, fake, 4, 2, 128, 128, 8, 0, 0, None,
                               None) == 1
    from gated_delta_rule_08_gb300.binding import _Epilogue
    epi = _Epilogue(0x1008, None, 1e-6)
    assert lib.kda_decode_multi(fake, fake, fake, fake, fake, fake, fake, None, fake, 4, 3, 2, 128, 128, 8, 0, 0, 0,
                                ctypes.byref(epi), None) == 1
    # checkpoints: no state buffer, interval < 1, misaligned buffer
    args = (fake, fake, fake, fake, fake, None, None, P(0x2000), None)
    tail = (1, 64, 1, 128, 128, 64, 0, 0, None, fake, 1 << 20, None)
    assert lib.kda_chunk_fwd_checkpoints(*args, None, 8, *tail) == 1
    assert lib.kda_chunk_fwd_checkpoints(*args, P(0x4000), 0, *tail) == 1
    assert lib.kda_chunk_fwd_checkpoints(*args, P(0x4004), 8, *tail) == 1
