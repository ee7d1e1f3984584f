"""CPU oracle of the QSA decode / MTP-verify step (test infrastructure only)."""
