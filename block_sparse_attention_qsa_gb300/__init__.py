"""QSA decode / MTP-verify step for GB300 (sm_103a).

Submodules:
  qsa    -- ctypes binding to the C-ABI library ``libqsa.so`` (loads on import
            and raises if the library is missing: there is no CPU fallback)
  synth  -- seeded synthetic inputs (random draws and storage formats only)
"""
