"""gMAGNUS-style SpGEMM C = A*B over CSR on one GB300 (sm_103a).

The compute path lives in the CUDA library ``libgm_spgemm.so`` behind a C ABI
(``include/gm_spgemm.h``); ``binding`` marshals torch tensors into it.
``inputs`` draws the seeded synthetic matrices.
"""
