"""CPU-side checks of the C ABI: the library loads, exports every declared symbol, and its NF4 table agrees with the oracle."""
import numpy as np

import layer_streamed_qlora_linear_b300 as sl
from oracle import nf4


def test_library_exports_every_header_symbol():
    lib = sl.lib()
    names = sl.header_functions()
    assert len(names) >= 15
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_code_table_match_oracle_bitwise():
    assert sl.sl_version() >= 10000
    t = np.array(sl.sl_nf4_code_table(), dtype=np.float32)
    assert np.array_equal(t.view(np.uint32), nf4.code_table().view(np.uint32))


def test_python_binding_declares_every_symbol():
    assert set(sl.header_functions()) <= set(sl._SIGS)
