"""The Python binding refuses tensors that the kernels would index out of bounds.

Every call passes one [batch, rows, cols] shape to the library, which indexes all
of the call's tensors with it, so a tensor of another size must be refused before
any pointer reaches the device.  The checks run before the device checks, so CPU
tensors exercise them here.
"""
import pytest
import torch

import newton_schulz_stacked_gb300 as nss

pytestmark = pytest.mark.filterwarnings("ignore")


def _bank(shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def test_step_refuses_tensors_of_another_size():
    sh = (2, 8, 16)
    bank, mant = _bank(sh), _bank(sh, torch.int16)
    mom = torch.zeros(sh, dtype=torch.float32)
    with pytest.raises(ValueError, match="grad has 255 elements, expected 256"):
        nss.muon_bank_step(bank, _bank((255,)), mom, mant, 0.02, 0.01, 0.95)
    with pytest.raises(ValueError, match="momentum"):
        nss.muon_bank_step(bank, _bank(sh), torch.zeros((2, 8, 15), dtype=torch.float32), mant, 0.02, 0.01, 0.95)
    with pytest.raises(ValueError, match="row_state has 15 elements, expected 16"):
        nss.normuon_bank_step(bank, _bank(sh), mom, mant, torch.zeros(15), 0.02, 0.01, 0.95)


def test_stages_refuse_tensors_of_another_size():
    sh = (2, 8, 16)
    with pytest.raises(ValueError, match="v has"):
        nss.mb_newton_schulz(_bank(sh), _bank((2, 8, 8)))
    with pytest.raises(ValueError, match="u has"):
        nss.mb_momentum(_bank(sh), torch.zeros(sh), _bank((1, 8, 16)), 0.95)
    with pytest.raises(ValueError, match="mantissa has"):
        nss.mb_update(_bank(sh), _bank((2, 16, 8, 2)), _bank(sh), 0.02, 0.01)


def test_multi_step_refuses_an_empty_bank_list_and_mismatched_banks():
    with pytest.raises(ValueError, match="no banks"):
        nss.muon_multi_step([], 0.02, 0.01, 0.95)
    sh = (3, 4, 4)
    bad = nss.BankState(_bank(sh), _bank(sh), torch.zeros(sh), _bank((3, 4, 3)))
    with pytest.raises(ValueError, match="mantissa"):
        nss.muon_multi_step([bad], 0.02, 0.01, 0.95)
